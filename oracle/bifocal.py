"""fp64 CPU oracle for causal bifocal-RoPE attention (Jet-Long).

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.  It
shares no code, table or constant with the CUDA path.

Sources (page title; section / equation):

  [D]  "Jet-Long: Efficient Long-Context Extension with Dynamic Bifocal RoPE",
       paper digest page, section "Method": the bifocal score S(q, k) (Eq. 1),
       the dynamic group size G and the alias map f (Eqs. 2-3), the KV-cache
       invariant with the correction offsets Delta_q, Delta_k (Eqs. 5-6) and
       the inclusion-exclusion prefill merge (Eq. 7).
  [P]  "Pith review of arXiv 2607.07740": the equation numbers above
       (Sections 3.1-3.3) and the statement that the construction is exact
       under standard RoPE composition (R_a R_b = R_{a+b}).
  [R]  RoFormer (cited by both pages): the rotary embedding R_p, a rotation
       of each coordinate pair by the angle p * omega_i.

Readings where the pages are silent, ambiguous or garbled:

  1. positions are 0-based, x in [0, L);
  2. in decode, L counts the cached tokens INCLUDING the new one, whose
     position is L-1;
  3. the cache holds keys already rotated at their absolute position;
  4. q-k == w0 is local ("<=" in Eq. 1);
  5. rotate-half pairing (x_i, x_{i+d/2}) with omega_i = theta^(-2i/d) and
     the RoFormer rotation [[cos, -sin], [sin, cos]];
  6. one softmax scale (default 1/sqrt(d)) for both branches;
  7. lse is the natural-log log-sum-exp of the scaled scores;
  8. GQA: query head h reads KV head h // (Hq // Hkv);
  9. one G for a whole prefill call, from the call's L;
 10. Eq. 7's passes: A = local window at absolute RoPE, B = every causal key
     at aliased RoPE, C = local window at aliased RoPE;
 11. ``round_rotated_qk=True`` rounds the rotated Q and K (both variants) to
     bf16 (round to nearest even), the operand precision of a bf16
     tensor-core kernel; P and everything else stay fp64.

Pins (all in ``tests/``, ``-m "not gpu"``):

  group_size         brute force: smallest g >= 1 with (L-1)//g < w_pretrained
  alias              integer identity f(x) = x + Delta(x), Delta <= 0
  rope_cos_sin       mpmath at 40 digits; additive angle R_a R_b = R_{a+b}
  rope_rotate        hand-derived values at d = 2 and d = 4 (pairing, sign)
  round_to_bf16      torch's float32 -> bfloat16 conversion
  bifocal_prefill    closed-form d = 2 golden table (tests/golden); G = 1 and
                     all-local both reduce to a textbook causal RoPE attention
                     written independently with complex numbers; Eq. 7
                     three-pass merge; V == 1 gives O == 1; remote scores are
                     shift-invariant by multiples of G.
  bifocal_decode     decode at length L equals prefill row L-1 on an unrounded
                     cache; V == 1.
  bifocal_prefill_chunk  with an unrounded cache equals the rows of
                     bifocal_prefill (additive angle); a one-token chunk
                     equals bifocal_decode on the same cache.
  bifocal_prefill_three_pass   agrees with bifocal_prefill (the two pin each
                     other: different algorithms for the same Eq. 1 result).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bifocal_prefill_chunk",
    "group_size",
    "alias",
    "rope_frequencies",
    "rope_cos_sin",
    "rope_rotate",
    "round_to_bf16",
    "bifocal_prefill",
    "bifocal_prefill_three_pass",
    "bifocal_decode",
]


# --------------------------------------------------------------------------
# Position mapping  [D, Method: "Dynamic group size"; P, Section 3.1, Eqs. 2-3]
# --------------------------------------------------------------------------

def group_size(L: int, w_pretrained: int) -> int:
    """G = max(1, ceil(L / w_pretrained)).

    [D, Method, Eq. 2]: the smallest integer that keeps every remote
    position inside the pretrained window.  L == 0 gives 1 (the max(1, .)).
    """
    L = int(L)
    w = int(w_pretrained)
    if L < 0 or w <= 0:
        raise ValueError(f"group_size: need L >= 0 and w_pretrained > 0, got {L}, {w}")
    return max(1, -(-L // w))


def alias(x, G: int):
    """f(x) = floor(x / G)  [D, Method, Eq. 3].  Works on ints and int arrays."""
    if isinstance(x, (int, np.integer)):
        return int(x) // int(G)
    return np.floor_divide(np.asarray(x, dtype=np.int64), int(G))


# --------------------------------------------------------------------------
# Rotary embedding  [R; D, Method: RoPE(x, p)]
# --------------------------------------------------------------------------

def rope_frequencies(d: int, theta: float) -> np.ndarray:
    """omega_i = theta^(-2i/d) for i = 0 .. d/2-1, fp64."""
    if d % 2:
        raise ValueError("head dim must be even")
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / d)


def rope_cos_sin(positions, d: int, theta: float):
    """cos and sin of n * omega_i for integer n (may be negative), fp64.

    The angle n * omega_i reaches 1.3e5 rad at n = 131071; forming it as one
    fp64 product loses about 1e-11 rad.  Instead R_n is built as the product
    of R_{2^j omega_i} over the set bits j of |n|: 2^j * omega_i is exact in
    binary floating point and libm reduces an exact argument correctly, so
    every factor is correct to rounding and the composition (angle-addition
    formulas) keeps the error near 1e-15.  R_{-n} is the transpose of R_n.
    Returns two arrays of shape positions.shape + (d/2,).
    """
    pos = np.asarray(positions, dtype=np.int64)
    omega = rope_frequencies(d, theta)
    mag = np.abs(pos)
    c = np.ones(pos.shape + (d // 2,), dtype=np.float64)
    s = np.zeros(pos.shape + (d // 2,), dtype=np.float64)
    nbits = int(mag.max()).bit_length() if mag.size else 0
    for j in range(nbits):
        ang = omega * float(2 ** j)
        cj, sj = np.cos(ang), np.sin(ang)
        bit = ((mag >> j) & 1).astype(bool)[..., None]
        c_new = c * cj - s * sj
        s_new = s * cj + c * sj
        c = np.where(bit, c_new, c)
        s = np.where(bit, s_new, s)
    s = np.where((pos < 0)[..., None], -s, s)
    return c, s


def _rotate(x: np.ndarray, c: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE with given cos/sin: pair (x_i, x_{i+d/2}) turns by the
    angle whose cos/sin are c_i, s_i (RoFormer rotation [[c, -s], [s, c]])."""
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_rotate(x, positions, theta: float) -> np.ndarray:
    """R_p x for x of shape [n, ..., d] and positions of shape [n]."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    c, s = rope_cos_sin(positions, d, theta)
    shape = (c.shape[0],) + (1,) * (x.ndim - 2) + (d // 2,)
    return _rotate(x, c.reshape(shape), s.reshape(shape))


def round_to_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value, ties to even.

    bf16 keeps 8 significant bits, so a value in [2^(e-1), 2^e) is rounded to
    a multiple of 2^(e-8); the exponent is clamped at bf16's smallest normal
    (2^-126) so that subnormals share the fixed quantum 2^-133.  The scaling
    by a power of two is exact and numpy's round() is half-to-even.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    quantum = np.ldexp(1.0, e - 8)
    return np.round(x / quantum) * quantum


# --------------------------------------------------------------------------
# Prefill  [D, Method: bifocal score, Eq. 1; masked causal softmax]
# --------------------------------------------------------------------------

def _softmax_rows(s: np.ndarray, vals: np.ndarray):
    """Row softmax of s (masked entries are -inf) applied to vals; returns
    (o, lse) with lse the natural-log log-sum-exp of each row."""
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=-1, keepdims=True)
    o = (p @ vals) / l
    return o, (m + np.log(l))[..., 0]


def _rows_for_head(rows, h: int, L: int) -> np.ndarray:
    if rows is None:
        return np.arange(L, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    return rows[h] if rows.ndim == 2 else rows


def bifocal_prefill(q, k, v, w0: int, w_pretrained: int, theta: float,
                    scale: float | None = None, round_rotated_qk: bool = False,
                    rows=None, row_chunk: int = 256):
    """Causal bifocal-RoPE attention over raw (pre-RoPE) q, k, v.

    For query position q and key position k <= q  [D, Method, Eq. 1]:
        local  (q - k <= w0):  s = scale * <R_q x_q, R_k x_k>
        remote (q - k >  w0):  s = scale * <R_f(q) x_q, R_f(k) x_k>
    with f(x) = floor(x / G) and G = group_size(L, w_pretrained)  [Eqs. 2-3];
    then an explicit masked causal softmax.

    q: [B, L, Hq, d]; k, v: [B, L, Hkv, d] (any real dtype; read as fp64).
    rows: None (every row) or query rows to evaluate, shape [n] or [Hq, n].
    Returns (o, lse): o [B, n, Hq, d], lse [B, Hq, n] in fp64 (n = L when
    rows is None).
    """
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    G = group_size(L, w_pretrained)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pos = np.arange(L, dtype=np.int64)
    fpos = alias(pos, G)
    # Every aliased position lies in [0, L), so one table serves both maps.
    cos_t, sin_t = rope_cos_sin(pos, d, theta)
    n_out = L if rows is None else np.asarray(rows).shape[-1]
    o_out = np.zeros((B, n_out, Hq, d), dtype=np.float64)
    lse_out = np.zeros((B, Hq, n_out), dtype=np.float64)
    rnd = round_to_bf16 if round_rotated_qk else (lambda a: a)
    for b in range(B):
        for hk in range(Hkv):
            xk = np.asarray(k[b, :, hk, :], dtype=np.float64)
            vk = np.asarray(v[b, :, hk, :], dtype=np.float64)
            k_abs = rnd(_rotate(xk, cos_t, sin_t))
            k_rem = rnd(_rotate(xk, cos_t[fpos], sin_t[fpos]))
            for h in range(hk * group, (hk + 1) * group):
                rh = _rows_for_head(rows, h, L)
                for c0 in range(0, rh.shape[0], row_chunk):
                    rc = rh[c0:c0 + row_chunk]
                    xq = np.asarray(q[b, rc, h, :], dtype=np.float64)
                    q_abs = rnd(_rotate(xq, cos_t[rc], sin_t[rc]))
                    q_rem = rnd(_rotate(xq, cos_t[fpos[rc]], sin_t[fpos[rc]]))
                    dist = rc[:, None] - pos[None, :]          # q - k
                    s_abs = q_abs @ k_abs.T
                    s_rem = q_rem @ k_rem.T
                    s = scale * np.where(dist <= w0, s_abs, s_rem)
                    s = np.where(dist < 0, -np.inf, s)
                    o, lse = _softmax_rows(s, vk)
                    o_out[b, c0:c0 + rc.shape[0], h, :] = o
                    lse_out[b, h, c0:c0 + rc.shape[0]] = lse
    return o_out, lse_out


def bifocal_prefill_three_pass(q, k, v, w0: int, w_pretrained: int, theta: float,
                               scale: float | None = None):
    """The pages' own prefill algorithm: three masked causal attentions merged
    by inclusion-exclusion with their log-sum-exp statistics
    [D, Method: "Inclusion-exclusion prefill", Eq. 7; P, Section 3.3].

      A: keys with q - k <= w0, absolute RoPE      -> (O_A, l_A)
      B: every causal key, aliased RoPE           -> (O_B, l_B)
      C: keys with q - k <= w0, aliased RoPE       -> (O_C, l_C)
      M = max(l_A, l_B, l_C),  W_X = exp(l_X - M)
      O = (W_A O_A + W_B O_B - W_C O_C) / (W_A + W_B - W_C)
      lse = M + log(W_A + W_B - W_C)

    Full L x L only (small inputs).  Same shapes as bifocal_prefill.
    """
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    group = Hq // Hkv
    G = group_size(L, w_pretrained)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pos = np.arange(L, dtype=np.int64)
    fpos = alias(pos, G)
    dist = pos[:, None] - pos[None, :]
    causal = dist >= 0
    window = causal & (dist <= w0)
    o_out = np.zeros((B, L, Hq, d))
    lse_out = np.zeros((B, Hq, L))
    for b in range(B):
        for h in range(Hq):
            hk = h // group
            xq = np.asarray(q[b, :, h, :], dtype=np.float64)
            xk = np.asarray(k[b, :, hk, :], dtype=np.float64)
            vk = np.asarray(v[b, :, hk, :], dtype=np.float64)
            s_abs = scale * (rope_rotate(xq, pos, theta) @ rope_rotate(xk, pos, theta).T)
            s_ali = scale * (rope_rotate(xq, fpos, theta) @ rope_rotate(xk, fpos, theta).T)
            o_a, l_a = _softmax_rows(np.where(window, s_abs, -np.inf), vk)
            o_b, l_b = _softmax_rows(np.where(causal, s_ali, -np.inf), vk)
            o_c, l_c = _softmax_rows(np.where(window, s_ali, -np.inf), vk)
            m = np.maximum(np.maximum(l_a, l_b), l_c)
            w_a, w_b, w_c = np.exp(l_a - m), np.exp(l_b - m), np.exp(l_c - m)
            den = w_a + w_b - w_c
            o_out[b, :, h, :] = (w_a[:, None] * o_a + w_b[:, None] * o_b
                                 - w_c[:, None] * o_c) / den[:, None]
            lse_out[b, h, :] = m + np.log(den)
    return o_out, lse_out


# --------------------------------------------------------------------------
# Chunked prefill against a cache  [D, Method: "KV cache invariant"]
# --------------------------------------------------------------------------

def bifocal_prefill_chunk(q, k, v, k_cache, P0: int, w0: int, w_pretrained: int, theta: float,
                          scale: float | None = None, round_rotated_qk: bool = False):
    """Queries of a chunk at positions P0 .. P0+C-1 against a cache of
    positions 0 .. P0-1 plus the chunk's own keys (causal).

    q: [B, C, Hq, d] raw chunk queries; k: [B, C, Hkv, d] raw chunk keys;
    v: [B, P0+C, Hkv, d] values of every position; k_cache: [B, >= P0, Hkv, d]
    holding R_j x_j for j < P0 as stored (read exactly, never modified).
    G = group_size(P0 + C, w_pretrained).  Cached keys take their aliased
    rotation through the correction R_{f(j) - j} applied to the stored key,
    the chunk's keys are rotated from raw; then the same piecewise score and
    masked causal softmax as bifocal_prefill.  ``round_rotated_qk`` rounds
    every rotated query and key that is not already a stored cache entry to
    bf16 (the tensor-core operands).  Returns (o [B, C, Hq, d], lse [B, Hq, C]).
    """
    B, C, Hq, d = q.shape
    Hkv = k.shape[2]
    group = Hq // Hkv
    Lt = P0 + C
    G = group_size(Lt, w_pretrained)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rnd = round_to_bf16 if round_rotated_qk else (lambda a: a)
    qpos = np.arange(P0, Lt, dtype=np.int64)
    kpos = np.arange(Lt, dtype=np.int64)
    cpos = np.arange(P0, dtype=np.int64)
    o_out = np.zeros((B, C, Hq, d))
    lse_out = np.zeros((B, Hq, C))
    dist = qpos[:, None] - kpos[None, :]
    for b in range(B):
        for hk in range(Hkv):
            cached = np.asarray(k_cache[b, :P0, hk, :], dtype=np.float64)
            xk = np.asarray(k[b, :, hk, :], dtype=np.float64)
            k_abs = np.concatenate([cached, rnd(rope_rotate(xk, qpos, theta))], axis=0)
            k_rem = np.concatenate([rnd(rope_rotate(cached, alias(cpos, G) - cpos, theta)),
                                    rnd(rope_rotate(xk, alias(qpos, G), theta))], axis=0)
            vk = np.asarray(v[b, :Lt, hk, :], dtype=np.float64)
            for h in range(hk * group, (hk + 1) * group):
                xq = np.asarray(q[b, :, h, :], dtype=np.float64)
                q_abs = rnd(rope_rotate(xq, qpos, theta))
                q_rem = rnd(rope_rotate(xq, alias(qpos, G), theta))
                s = scale * np.where(dist <= w0, q_abs @ k_abs.T, q_rem @ k_rem.T)
                s = np.where(dist < 0, -np.inf, s)
                o, lse = _softmax_rows(s, vk)
                o_out[b, :, h, :] = o
                lse_out[b, h, :] = lse
    return o_out, lse_out


# --------------------------------------------------------------------------
# Decode  [D, Method: "KV cache invariant", Eqs. 5-6]
# --------------------------------------------------------------------------

def bifocal_decode(q, k_cache, v_cache, L: int, w0: int, w_pretrained: int,
                   theta: float, scale: float | None = None):
    """One new query token at position L-1 against an absolute-position cache.

    q: [B, Hq, d] raw (pre-RoPE); k_cache: [B, Lcap, Hkv, d] holding R_j x_j
    (keys rotated at their absolute position j); v_cache: [B, Lcap, Hkv, d].
    Keys j in [0, L) are read; the cache itself is never modified.

      G = group_size(L, w_pretrained), f(x) = floor(x / G), qp = L - 1
      local  (qp - j <= w0):  s_j = scale * <R_qp x_q, K_j>
      remote (qp - j >  w0):  s_j = scale * <R_f(qp) x_q, R_(f(j)-j) K_j>

    The remote key is corrected on the fly by Delta_k = f(j) - j
    (R_Delta R_j = R_f(j), the additive-angle property) [D, Method; P, 3.2].
    Returns (o [B, Hq, d], lse [B, Hq]) in fp64.
    """
    B, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    group = Hq // Hkv
    if not (1 <= L <= k_cache.shape[1]):
        raise ValueError("need 1 <= L <= Lcap")
    G = group_size(L, w_pretrained)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qp = L - 1
    j = np.arange(L, dtype=np.int64)
    delta_k = alias(j, G) - j
    c_d, s_d = rope_cos_sin(delta_k, d, theta)
    local = (qp - j) <= w0
    o_out = np.zeros((B, Hq, d))
    lse_out = np.zeros((B, Hq))
    for b in range(B):
        for hk in range(Hkv):
            kc = np.asarray(k_cache[b, :L, hk, :], dtype=np.float64)
            vc = np.asarray(v_cache[b, :L, hk, :], dtype=np.float64)
            k_corr = _rotate(kc, c_d, s_d)
            for h in range(hk * group, (hk + 1) * group):
                xq = np.asarray(q[b, h, :], dtype=np.float64)[None, :]
                q_abs = rope_rotate(xq, [qp], theta)[0]
                q_rem = rope_rotate(xq, [alias(qp, G)], theta)[0]
                s = scale * np.where(local, kc @ q_abs, k_corr @ q_rem)
                o, lse = _softmax_rows(s[None, :], vc)
                o_out[b, h, :] = o[0]
                lse_out[b, h] = lse[0]
    return o_out, lse_out
