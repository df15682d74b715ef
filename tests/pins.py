"""Pins for the fp64 oracle: checks against what the Jet-Long pages and the
mathematics fix, independent of the oracle's own formulas.

Every pin takes the oracle module as ``orc`` so that ``test_oracle_mutations``
can run the same pins against deliberately broken copies of the oracle and
show that each plausible mistake is caught.  Each pin raises AssertionError
on failure.

Sources: "Jet-Long: Efficient Long-Context Extension with Dynamic Bifocal
RoPE" (paper digest page), section "Method" (Eq. 1 bifocal score, Eqs. 2-3
G and f, Eqs. 5-6 correction rotation, Eq. 7 inclusion-exclusion merge);
RoFormer for R_p.
"""

from __future__ import annotations

import math
import os

import mpmath
import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers

def textbook_causal_rope_attention(q, k, v, theta, scale):
    """Ordinary causal RoPE attention, written independently of the oracle:
    torch fp64, RoPE as multiplication of the complex pairs
    (x_i + i x_{i+d/2}) by exp(i p omega_i), torch.softmax / logsumexp.
    q, k, v: [L, d] (one head).  Returns (o [L, d], lse [L])."""
    q = torch.as_tensor(np.asarray(q, dtype=np.float64))
    k = torch.as_tensor(np.asarray(k, dtype=np.float64))
    v = torch.as_tensor(np.asarray(v, dtype=np.float64))
    L, d = q.shape
    h = d // 2
    inv = torch.tensor(float(theta), dtype=torch.float64) ** (
        -torch.arange(h, dtype=torch.float64) * 2.0 / d)
    ang = torch.arange(L, dtype=torch.float64)[:, None] * inv[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)
    qc = torch.complex(q[:, :h], q[:, h:]) * rot
    kc = torch.complex(k[:, :h], k[:, h:]) * rot
    s = (qc.real @ kc.real.T + qc.imag @ kc.imag.T) * scale
    mask = torch.triu(torch.ones(L, L, dtype=torch.bool), diagonal=1)
    s = s.masked_fill(mask, float("-inf"))
    return (torch.softmax(s, dim=-1) @ v).numpy(), torch.logsumexp(s, dim=-1).numpy()


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def read_golden_angles(name="closed_form_d2.txt"):
    meta, rows = {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("q "):
                head, tail = line.split(":")
                rows[int(head.split()[1])] = [int(t) for t in tail.split()]
            else:
                key, val = line.split()
                meta[key] = int(val)
    return meta, rows


# ---------------------------------------------------------------- pins

def pin_group_size_bruteforce(orc):
    """G is the smallest integer g >= 1 with floor((L-1)/g) < w_pretrained
    (all positions 0..L-1 alias into the pretrained window); L = 0 gives 1."""
    def brute(L, w):
        if L == 0:
            return 1
        g = 1
        while (L - 1) // g >= w:
            g += 1
        return g
    for w in (1, 2, 3, 7, 64, 1000, 32768):
        Ls = list(range(0, min(40 * w, 3000))) + [w - 1, w, w + 1, 2 * w, 2 * w + 1,
                                                  4 * w, 4 * w + 1, 50 * w - 1]
        for L in Ls:
            if L < 0:
                continue
            assert orc.group_size(L, w) == brute(L, w), (L, w)
    # the five workloads' lengths
    for L, w, g in ((256, 64, 4), (32768, 32768, 1), (65536, 32768, 2), (131072, 32768, 4),
                    (32767, 32768, 1), (32769, 32768, 2), (65537, 32768, 3)):
        assert orc.group_size(L, w) == g


def pin_alias_floor(orc):
    """f(x) = floor(x/G): 0 <= x - G f(x) < G; f(x + cG) = f(x) + c;
    Delta(x) = f(x) - x <= 0."""
    for G in (1, 2, 3, 4, 7):
        x = np.arange(0, 5000, dtype=np.int64)
        f = np.asarray(orc.alias(x, G))
        r = x - G * f
        assert np.all((r >= 0) & (r < G))
        assert np.array_equal(np.asarray(orc.alias(x + 5 * G, G)), f + 5)
        assert np.all(f - x <= 0)


def pin_rope_mpmath(orc):
    """cos/sin(n * omega_i) against mpmath at 40 digits, for the oracle's own
    fp64 omega_i (converted exactly); omega_i against theta^(-2i/d)."""
    mpmath.mp.dps = 40
    for d, theta in ((128, 1e6), (64, 1e4), (16, 500.0)):
        om = orc.rope_frequencies(d, theta)
        for i in range(d // 2):
            ref = mpmath.power(mpmath.mpf(theta), mpmath.mpf(-2 * i) / d)
            assert abs(float((mpmath.mpf(float(om[i])) - ref) / ref)) < 4e-16
        pos = np.array([0, 1, 2, 3, 1000, 32767, 32768, 65535, 98303, 131071, -1, -98304,
                        -32767], dtype=np.int64)
        c, s = orc.rope_cos_sin(pos, d, theta)
        for a, n in enumerate(pos):
            for i in range(0, d // 2, max(1, d // 32)):
                ang = mpmath.mpf(int(n)) * mpmath.mpf(float(om[i]))
                assert abs(c[a, i] - float(mpmath.cos(ang))) < 3e-15, (n, i)
                assert abs(s[a, i] - float(mpmath.sin(ang))) < 3e-15, (n, i)


def pin_rope_hand_values(orc):
    """RoFormer rotation with rotate-half pairing, values derived by hand.
    d = 2: R_p (1,0) = (cos p, sin p), R_p (0,1) = (-sin p, cos p).
    d = 4, theta = 100: omega = (1, 0.1); pairs are (x0, x2) and (x1, x3)."""
    for p in (0, 1, 3, 17):
        out = orc.rope_rotate(np.array([[1.0, 0.0], [0.0, 1.0]])[None], [p], 10000.0)[0]
        assert np.allclose(out[0], [math.cos(p), math.sin(p)], atol=1e-15, rtol=0)
        assert np.allclose(out[1], [-math.sin(p), math.cos(p)], atol=1e-15, rtol=0)
    eye = np.eye(4)[None]                       # [1, 4 rows, 4]
    out = orc.rope_rotate(eye, [3], 100.0)[0]
    c3, s3 = -0.9899924966004454, 0.1411200080598672     # cos 3, sin 3
    c03, s03 = 0.955336489125606, 0.29552020666133955    # cos 0.3, sin 0.3
    expect = np.array([[c3, 0.0, s3, 0.0],
                       [0.0, c03, 0.0, s03],
                       [-s3, 0.0, c3, 0.0],
                       [0.0, -s03, 0.0, c03]])
    assert np.allclose(out, expect, atol=2e-15, rtol=0), out


def pin_additive_angle(orc):
    """R_{f(k)-k} (R_k x) == R_{f(k)} x to 1e-12 for k up to 131071
    (the additive-angle property behind the cache correction, Eqs. 5-6)."""
    k = np.array([0, 1, 4095, 4096, 32767, 32768, 65537, 98303, 131070, 131071])
    x = _rand((k.size, 2, 128), 7)
    for G in (2, 3, 4):
        f = orc.alias(k, G)
        lhs = orc.rope_rotate(orc.rope_rotate(x, k, 1e6), f - k, 1e6)
        rhs = orc.rope_rotate(x, f, 1e6)
        assert np.abs(lhs - rhs).max() <= 1e-12


def pin_round_to_bf16(orc):
    """Round-to-nearest-even bf16 equals torch's float32 -> bfloat16 cast,
    including exact ties and tiny/huge magnitudes."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-30,
                        rng.standard_normal(2000) * 1e30]).astype(np.float32)
    base = torch.from_numpy(rng.standard_normal(4000).astype(np.float32)).to(torch.bfloat16)
    b = base.view(torch.int16).numpy().astype(np.int64) & 0xFFFF
    ties = ((b << 16) | 0x8000).astype(np.uint32).view(np.float32)       # exactly half-way
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = orc.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(ref, got)


def pin_closed_form_golden(orc):
    """Hand-derived angles (tests/golden/closed_form_d2.txt): d = 2, raw q-rows
    e1, raw k-rows e1 (score cos a) or e2 (score sin a), value row k = (k, 1);
    then O[q] = (sum_k k w_k / sum_k w_k, 1) and lse = log sum_k w_k with
    w_k = exp(scale * score), scale = 1/sqrt(2)."""
    meta, rows = read_golden_angles()
    L, wp, w0 = meta["L"], meta["w_pretrained"], meta["w0"]
    assert orc.group_size(L, wp) == meta["G"]
    q = np.zeros((1, L, 1, 2)); q[..., 0] = 1.0
    v = np.zeros((1, L, 1, 2)); v[0, :, 0, 0] = np.arange(L); v[..., 1] = 1.0
    for kind, fn in (("cos", math.cos), ("sin", math.sin)):
        k = np.zeros((1, L, 1, 2))
        k[..., 0 if kind == "cos" else 1] = 1.0
        o, lse = orc.bifocal_prefill(q, k, v, w0, wp, 10000.0)
        for qq, angles in rows.items():
            w = [math.exp(fn(a) / math.sqrt(2.0)) for a in angles]
            o0 = sum(kk * wk for kk, wk in enumerate(w)) / sum(w)
            assert abs(o[0, qq, 0, 0] - o0) < 1e-12, (kind, qq)
            assert abs(o[0, qq, 0, 1] - 1.0) < 1e-12
            assert abs(lse[0, 0, qq] - math.log(sum(w))) < 1e-12, (kind, qq)


def pin_g1_is_textbook(orc):
    """L <= w_pretrained => G = 1 => ordinary causal RoPE attention
    [digest, Method: "reduces exactly to the base model"]."""
    for (L, wp, w0, d, theta) in ((200, 256, 16, 32, 1e4), (64, 64, 0, 16, 1e6), (33, 40, 5, 8, 500.0)):
        Hq, Hkv = 4, 2
        q, k, v = _rand((1, L, Hq, d), 1), _rand((1, L, Hkv, d), 2), _rand((1, L, Hkv, d), 3)
        o, lse = orc.bifocal_prefill(q, k, v, w0, wp, theta)
        for h in range(Hq):
            ot, lt = textbook_causal_rope_attention(q[0, :, h], k[0, :, h // 2], v[0, :, h // 2],
                                                    theta, 1 / math.sqrt(d))
            assert np.abs(o[0, :, h] - ot).max() <= 1e-12
            assert np.abs(lse[0, h] - lt).max() <= 1e-12


def pin_all_local_is_textbook(orc):
    """w0 >= L-1: every pair is local, so any G gives causal RoPE attention."""
    for (L, wp, w0) in ((100, 16, 99), (100, 16, 150), (57, 7, 56)):
        d = 16
        q, k, v = _rand((1, L, 2, d), 4), _rand((1, L, 1, d), 5), _rand((1, L, 1, d), 6)
        assert orc.group_size(L, wp) > 1
        o, lse = orc.bifocal_prefill(q, k, v, w0, wp, 1e4)
        for h in range(2):
            ot, lt = textbook_causal_rope_attention(q[0, :, h], k[0, :, 0], v[0, :, 0], 1e4,
                                                    1 / math.sqrt(d))
            assert np.abs(o[0, :, h] - ot).max() <= 1e-12
            assert np.abs(lse[0, h] - lt).max() <= 1e-12


def pin_three_pass_merge(orc):
    """Eq. 7's three-pass inclusion-exclusion merge equals the direct masked
    softmax over the piecewise score (tiny inputs, fp64)."""
    for L in (1, 2, 17, 64):
        for G in (1, 2, 3, 4):
            wp = max(1, -(-L // G))
            if orc.group_size(L, wp) != G:
                continue
            for w0 in (0, 1, 5, L):
                q, k, v = _rand((1, L, 2, 8), L + G), _rand((1, L, 1, 8), 2 * L + G), _rand((1, L, 1, 8), 3)
                o1, l1 = orc.bifocal_prefill(q, k, v, w0, wp, 1e4)
                o2, l2 = orc.bifocal_prefill_three_pass(q, k, v, w0, wp, 1e4)
                assert np.abs(o1 - o2).max() <= 1e-12, (L, G, w0)
                assert np.abs(l1 - l2).max() <= 1e-12, (L, G, w0)


def pin_decode_equals_prefill_row(orc):
    """Decode at length L' on a cache holding R_j x_j (unrounded) equals the
    last row of a prefill over the first L' tokens (same G); the cache is
    read, never rewritten [digest, Method: "KV cache invariant"]."""
    Lmax, Hq, Hkv, d, wp, w0, theta = 40, 4, 2, 16, 10, 5, 1e4
    q, k, v = _rand((1, Lmax, Hq, d), 11), _rand((1, Lmax, Hkv, d), 12), _rand((1, Lmax, Hkv, d), 13)
    pos = np.arange(Lmax)
    cache_k = orc.rope_rotate(k[0], pos, theta)[None]
    before = cache_k.copy()
    for Lp in (1, 2, 6, 7, 10, 11, 21, 31, 40):
        od, ld = orc.bifocal_decode(q[:, Lp - 1], cache_k, v, Lp, w0, wp, theta)
        op, lp = orc.bifocal_prefill(q[:, :Lp], k[:, :Lp], v[:, :Lp], w0, wp, theta)
        assert np.abs(od[0] - op[0, Lp - 1]).max() <= 1e-12, Lp
        assert np.abs(ld[0] - lp[0, :, Lp - 1]).max() <= 1e-12, Lp
    assert np.array_equal(before, cache_k)


def pin_values_one(orc):
    """V == 1 gives O == 1 (probabilities sum to one), prefill and decode."""
    L, d = 50, 8
    q, k = _rand((1, L, 2, d), 21), _rand((1, L, 1, d), 22)
    v = np.ones((1, L, 1, d))
    o, _ = orc.bifocal_prefill(q, k, v, 3, 12, 1e4)
    assert np.abs(o - 1).max() <= 1e-14
    od, _ = orc.bifocal_decode(q[:, -1], k, v, L, 3, 12, 1e4)
    assert np.abs(od - 1).max() <= 1e-14


def pin_remote_shift_invariance(orc):
    """A remote score depends only on f(q) - f(k): shifting both positions by a
    multiple of G leaves <R_f(q) x, R_f(k) y> unchanged."""
    x, y = _rand((1, 64), 31), _rand((1, 64), 32)
    G = 3
    for (qp, kp) in ((100, 7), (90, 40), (2000, 3)):
        ref = None
        for c in (0, 1, 5, 400):
            a = orc.rope_rotate(x, [orc.alias(qp + c * G, G)], 1e4)
            b = orc.rope_rotate(y, [orc.alias(kp + c * G, G)], 1e4)
            val = float((a * b).sum())
            ref = val if ref is None else ref
            assert abs(val - ref) <= 1e-12


def pin_sampled_rows(orc):
    """Evaluating selected rows gives the full result's rows (to BLAS
    summation-order rounding)."""
    L = 90
    q, k, v = _rand((1, L, 2, 8), 41), _rand((1, L, 1, 8), 42), _rand((1, L, 1, 8), 43)
    o, lse = orc.bifocal_prefill(q, k, v, 4, 30, 1e4)
    rows = np.array([[0, 5, 89, 33], [1, 2, 60, 31]])
    os_, ls_ = orc.bifocal_prefill(q, k, v, 4, 30, 1e4, rows=rows, row_chunk=3)
    for h in range(2):
        assert np.abs(os_[0, :, h] - o[0, rows[h], h]).max() <= 1e-14
        assert np.abs(ls_[0, h] - lse[0, h, rows[h]]).max() <= 1e-14


def pin_chunk_equals_prefill_rows(orc):
    """A chunk against an unrounded cache (R_j x_j in fp64) equals the rows of
    a prefill over all positions so far (same G): the correction rotation
    R_{f(j)-j} R_j = R_{f(j)} (additive angle, "KV cache invariant")."""
    L, Hq, Hkv, d, wp, w0, theta = 60, 4, 2, 16, 17, 5, 1e4
    q, k, v = _rand((1, L, Hq, d), 51), _rand((1, L, Hkv, d), 52), _rand((1, L, Hkv, d), 53)
    for P0, C in ((0, 60), (20, 40), (33, 1), (59, 1), (1, 59)):
        Lt = P0 + C
        cache = orc.rope_rotate(k[0, :P0], np.arange(P0), theta)[None] if P0 else np.zeros((1, 0, Hkv, d))
        oc, lc = orc.bifocal_prefill_chunk(q[:, P0:Lt], k[:, P0:Lt], v, cache, P0, w0, wp, theta)
        op, lp = orc.bifocal_prefill(q[:, :Lt], k[:, :Lt], v[:, :Lt], w0, wp, theta)
        assert np.abs(oc - op[:, P0:Lt]).max() <= 1e-12, (P0, C)
        assert np.abs(lc - lp[:, :, P0:Lt]).max() <= 1e-12, (P0, C)


def pin_one_token_chunk_is_decode(orc):
    """A one-token chunk against a stored (bf16-rounded) cache equals decode
    on the same cache with the token's own rotated key appended."""
    L, Hq, Hkv, d, wp, w0, theta = 45, 4, 1, 16, 10, 3, 1e4
    q, k, v = _rand((1, L, Hq, d), 61), _rand((1, L, Hkv, d), 62), _rand((1, L, Hkv, d), 63)
    cache = orc.round_to_bf16(orc.rope_rotate(k[0], np.arange(L), theta))[None]
    P0 = L - 1
    oc, lc = orc.bifocal_prefill_chunk(q[:, P0:], k[:, P0:], v, cache, P0, w0, wp, theta)
    full_cache = cache.copy()
    full_cache[0, P0] = orc.rope_rotate(k[0, P0:], [P0], theta)[0]
    od, ld = orc.bifocal_decode(q[:, P0], full_cache, v, L, w0, wp, theta)
    assert np.abs(oc[:, 0] - od).max() <= 1e-12
    assert np.abs(lc[:, :, 0] - ld).max() <= 1e-12


ALL_PINS = [
    pin_group_size_bruteforce,
    pin_alias_floor,
    pin_rope_mpmath,
    pin_rope_hand_values,
    pin_additive_angle,
    pin_round_to_bf16,
    pin_closed_form_golden,
    pin_g1_is_textbook,
    pin_all_local_is_textbook,
    pin_three_pass_merge,
    pin_decode_equals_prefill_row,
    pin_values_one,
    pin_remote_shift_invariance,
    pin_sampled_rows,
    pin_chunk_equals_prefill_rows,
    pin_one_token_chunk_is_decode,
]
