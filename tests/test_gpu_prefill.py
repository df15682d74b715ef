"""Prefill parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases are compared element by element on every row; the 32K, 64K and
128K workloads on 512 seeded rows per query head (tests/sampling.py).  The
LSE is judged against the oracle mode that rounds the rotated Q and K to
bf16 (the tensor cores' operand precision); O against both modes."""

import math

import numpy as np
import pytest

import oracle
from bifocal_rope_extension_causal_b300 import synth, workloads as W
from gpu_common import assert_close, to_np
from sampling import oracle_prefill_rows, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jl():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bifocal_rope_extension_causal_b300 as mod
    from bifocal_rope_extension_causal_b300 import build
    build.build()
    return mod


def run_gpu(jl, q, k, v, w0, wp, theta, k_rot=False):
    import torch
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    krot = torch.empty_like(kd) if k_rot else None
    o, lse = jl.prefill(qd, kd, vd, w0, wp, theta, k_rot_out=krot)
    jl.device_status()
    return o, lse, krot


def full_check(jl, L, Hq, Hkv, d, wp, w0, theta, seed, B=1):
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, seed, B=B)
    o, lse, _ = run_gpu(jl, q, k, v, w0, wp, theta)
    qn, kn, vn = (x.float().numpy() for x in (q, k, v))
    o_r, l_r = oracle.bifocal_prefill(qn, kn, vn, w0, wp, theta, round_rotated_qk=True)
    o_p, _ = oracle.bifocal_prefill(qn, kn, vn, w0, wp, theta)
    og, lg = to_np(o), to_np(lse)
    tag = f"L={L} Hq={Hq} Hkv={Hkv} d={d} wp={wp} w0={w0} B={B}"
    assert_close(og, lg, o_r, l_r, tag + " (rounded oracle)")
    err = np.abs(og - o_p)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, tag + " (plain oracle)"


def test_tiny_workload(jl):
    w = W.TINY
    assert jl.group_size(w.L, w.w_pretrained) == 4
    full_check(jl, w.L, w.Hq, w.Hkv, w.d, w.w_pretrained, w.w0, w.theta, w.index)


@pytest.mark.parametrize("L,Hq,Hkv,d,wp,w0", [
    (1, 2, 1, 64, 64, 16),        # one row
    (2, 2, 2, 128, 1, 0),         # G = 2, w0 = 0
    (63, 4, 2, 64, 16, 5),        # ragged tail, G = 4
    (65, 4, 1, 128, 16, 0),       # one row past a tile, w0 = 0 (all remote but the diagonal)
    (129, 8, 2, 128, 40, 7),      # G = 4, three tiles, ragged
    (200, 4, 4, 64, 256, 16),     # G = 1: plain causal RoPE attention
    (300, 2, 1, 128, 50, 299),    # w0 >= L-1: all local at G = 6
    (333, 6, 2, 128, 37, 100),    # G = 10, straddle band across several tiles
    (512, 4, 2, 128, 128, 64),    # tile-aligned, straddles aligned with tiles
])
def test_small_shapes(jl, L, Hq, Hkv, d, wp, w0):
    full_check(jl, L, Hq, Hkv, d, wp, w0, 1e4, seed=L + 7 * w0)


@pytest.mark.parametrize("L,Hq,Hkv,d,wp,w0", [
    (5000, 16, 2, 128, 1700, 700),   # G = 3, GQA group 8, ragged, band across many tiles
    (4096, 4, 2, 64, 2048, 1000),    # d = 64, G = 2, multi-tile straddles
    (3000, 4, 1, 128, 800, 0),       # w0 = 0 over many tiles, G = 4
    (2304, 8, 8, 128, 300, 2303),    # every pair local at G = 8
])
def test_mid_sizes(jl, L, Hq, Hkv, d, wp, w0):
    full_check(jl, L, Hq, Hkv, d, wp, w0, 1e6, seed=L + w0)


@pytest.mark.parametrize("L,Hq,Hkv,wp,w0,B", [
    (65, 4, 1, 16, 0, 1),         # one row past a tile, all remote but the diagonal
    (129, 8, 2, 40, 7, 1),        # G = 4, ragged, three tiles
    (512, 4, 2, 128, 64, 1),      # tile-aligned straddles
    (3000, 4, 1, 800, 0, 1),      # w0 = 0 over many tiles, G = 4
    (2304, 8, 8, 300, 2303, 1),   # every pair local at G = 8
    (1000, 16, 2, 300, 100, 1),   # GQA group 8, G = 4
    (300, 4, 2, 100, 30, 2),      # batch of two, G = 3
])
def test_cta_pair_kernel_matches_oracle(jl, L, Hq, Hkv, wp, w0, B):
    """The CTA-pair attention kernel (the A/B counterpart of the default
    kernel, head dim 128) after jl_bifocal_rope, against the oracle."""
    import ctypes
    import torch
    from bifocal_rope_extension_causal_b300 import _capi
    d, theta = 128, 1e6
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, L + w0, B=B)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device="cuda")
    nbytes = jl.prefill_workspace_size(B, L, Hq, Hkv, d, wp)
    ws = jl.alloc_workspace(nbytes, qd.device)
    lib, P = _capi.load(), ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    _capi.check(lib.jl_bifocal_rope(P(qd.data_ptr()), P(kd.data_ptr()), B, L, Hq, Hkv, d, wp, theta, None,
                                    P(ws.data_ptr()), nbytes, stream))
    _capi.check(lib.jl_bifocal_attention_cta_pair(P(vd.data_ptr()), P(o.data_ptr()), P(lse.data_ptr()), B, L, Hq,
                                                  Hkv, d, w0, wp, 0.0, P(ws.data_ptr()), nbytes, stream))
    jl.device_status()
    qn, kn, vn = (x.float().numpy() for x in (q, k, v))
    o_r, l_r = oracle.bifocal_prefill(qn, kn, vn, w0, wp, theta, round_rotated_qk=True)
    o_p, _ = oracle.bifocal_prefill(qn, kn, vn, w0, wp, theta)
    og, lg = to_np(o), to_np(lse)
    tag = f"cta pair L={L} Hq={Hq} Hkv={Hkv} wp={wp} w0={w0} B={B}"
    assert_close(og, lg, o_r, l_r, tag + " (rounded oracle)")
    err = np.abs(og - o_p)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, tag + " (plain oracle)"


def test_batch_of_two(jl):
    full_check(jl, 150, 4, 2, 128, 40, 10, 1e6, seed=5, B=2)


def test_k_rot_out_is_the_absolute_rotation(jl):
    """k_rot_out holds R_k x_k (the cache form): exactly the oracle's rotation
    rounded to bf16, bit for bit."""
    L, Hq, Hkv, d = 96, 2, 2, 128
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, 11)
    _, _, krot = run_gpu(jl, q, k, v, 8, 32, 1e6, k_rot=True)
    ref = oracle.round_to_bf16(oracle.rope_rotate(k[0].float().numpy(), np.arange(L), 1e6))
    assert np.array_equal(to_np(krot)[0], ref)


@pytest.mark.parametrize("L,Hq,Hkv,d,wp,theta", [
    (4096, 8, 4, 128, 1024, 1e6),    # G = 4
    (3000, 4, 2, 64, 700, 1e4),      # G = 5, d = 64
    (1050000, 1, 1, 64, 300000, 1e6),  # positions past 2^20: all three table levels
])
def test_rotated_operands_are_exactly_rounded(jl, L, Hq, Hkv, d, wp, theta):
    """The rotated operands in the workspace (Q and K at absolute and aliased
    positions) equal the oracle's exact rotation rounded to bf16, bit for bit:
    the kernel's rounding decisions are those of the exact values."""
    import torch
    q, k, _ = synth.prefill_inputs(L, Hq, Hkv, d, 5)
    qd, kd = q.cuda(), k.cuda()
    nbytes = jl.prefill_workspace_size(1, L, Hq, Hkv, d, wp)
    ws = jl.alloc_workspace(nbytes, "cuda")
    jl.check(jl.load().jl_bifocal_rope(
        jl._ptr(qd), jl._ptr(kd), 1, L, Hq, Hkv, d, wp, theta, None, jl._ptr(ws), nbytes,
        jl._stream_ptr(None)))
    torch.cuda.synchronize()
    G = jl.group_size(L, wp)
    assert G > 1

    def part(off, H):
        n = H * L * d * 2
        t = ws[off:off + n].view(torch.bfloat16).view(H, L, d)
        return to_np(t), off + (n + 255) // 256 * 256

    qa, off = part(0, Hq)
    ka, off = part(off, Hkv)
    qr, off = part(off, Hq)
    kr, off = part(off, Hkv)
    pos = np.arange(L)
    fpos = pos // G
    for name, got, x, p in (("Q_abs", qa, q, pos), ("K_abs", ka, k, pos), ("Q_rem", qr, q, fpos),
                            ("K_rem", kr, k, fpos)):
        xs = x[0].float().numpy()  # [L, H, d]
        ref = oracle.round_to_bf16(oracle.rope_rotate(xs, p, theta)).transpose(1, 0, 2)
        bad = int((got != ref).sum())
        assert bad == 0, f"{name}: {bad} of {ref.size} elements differ from the exactly rounded rotation"


def test_values_one_gives_ones(jl):
    import torch
    L, Hq, Hkv, d = 257, 4, 2, 128
    q, k, _ = synth.prefill_inputs(L, Hq, Hkv, d, 3)
    v = torch.ones(1, L, Hkv, d, dtype=torch.bfloat16)
    o, _, _ = run_gpu(jl, q, k, v, 20, 64, 1e4)
    assert np.abs(to_np(o) - 1.0).max() <= 2.0 ** -8


def sampled_check(jl, w, n_rows=512):
    q, k, v = synth.prefill_inputs(w.L, w.Hq, w.Hkv, w.d, w.index)
    o, lse, _ = run_gpu(jl, q, k, v, w.w0, w.w_pretrained, w.theta)
    G = jl.group_size(w.L, w.w_pretrained)
    rows = np.stack([sample_rows(w.L, w.w0, w.w_pretrained, G, n_rows, 1000 * w.index + h)
                     for h in range(w.Hq)])
    og = np.stack([to_np(o[0, rows[h], h]) for h in range(w.Hq)], axis=1)[None]
    lg = np.stack([to_np(lse[0, h, rows[h]]) for h in range(w.Hq)])[None]
    del o, lse
    qn, kn, vn = (x.float().numpy() for x in (q, k, v))
    o_r, l_r = oracle_prefill_rows(qn, kn, vn, w.w0, w.w_pretrained, w.theta, rows, True)
    return assert_close(og, lg, o_r, l_r, w.name)


@pytest.mark.parametrize("w", [W.NATIVE_32K, W.EXT_64K, W.EXT_128K], ids=["32K", "64K", "128K"])
def test_full_size_sampled_rows(jl, w):
    sampled_check(jl, w)


def test_native_window_equals_plain_rope_attention(jl):
    """G = 1 (L = w_pretrained): every sampled row equals ordinary causal RoPE
    attention -- the oracle at w0 = L (all local) is that attention."""
    w = W.NATIVE_32K
    q, k, v = synth.prefill_inputs(w.L, w.Hq, w.Hkv, w.d, w.index)
    o, lse, _ = run_gpu(jl, q, k, v, w.w0, w.w_pretrained, w.theta)
    rows = np.stack([sample_rows(w.L, w.w0, w.w_pretrained, 1, 64, 77 + h) for h in range(w.Hq)])
    og = np.stack([to_np(o[0, rows[h], h]) for h in range(w.Hq)], axis=1)[None]
    lg = np.stack([to_np(lse[0, h, rows[h]]) for h in range(w.Hq)])[None]
    qn, kn, vn = (x.float().numpy() for x in (q, k, v))
    o_r, l_r = oracle_prefill_rows(qn, kn, vn, w.L, w.w_pretrained, w.theta, rows, True)
    assert_close(og, lg, o_r, l_r, "native window vs plain causal RoPE attention")
