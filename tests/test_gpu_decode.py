"""Decode parity: the CUDA split-K decode (through the C ABI) against the fp64
oracle, on the whole key range.  The cache is checksummed before and after
every step: it is read, never rewritten, while G crosses 1 -> 2 -> 3 -> 4."""

import numpy as np
import pytest

import oracle
from bifocal_rope_extension_causal_b300 import synth, workloads as W
from gpu_common import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jl():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bifocal_rope_extension_causal_b300 as mod
    from bifocal_rope_extension_causal_b300 import build
    build.build()
    return mod


def check_decode(jl, kc, vc, q, L, w0, wp, theta, tag):
    o, lse = jl.decode(q.cuda() if not q.is_cuda else q, kc, vc, L, w0, wp, theta)
    jl.device_status()
    o_ref, l_ref = oracle.bifocal_decode(q.float().cpu().numpy(), kc[:, :L].float().cpu().numpy(),
                                         vc[:, :L].float().cpu().numpy(), L, w0, wp, theta)
    return assert_close(to_np(o), to_np(lse), o_ref, l_ref, tag)


def test_decode_workload_cache_invariant(jl):
    """The decode workload: one cache, lengths 32767, 32769, 65537, 131072
    (G = 1, 2, 3, 4), the cache bytes unchanged after every step."""
    import torch
    w = W.DECODE
    kc, vc, qs = synth.decode_inputs(w.Lcap, w.Hq, w.Hkv, w.d, w.index, len(w.lengths))
    kc, vc = kc.cuda(), vc.cuda()
    sums = (kc.view(torch.int16).long().sum().item(), vc.view(torch.int16).long().sum().item())
    for step, L in enumerate(w.lengths):
        G = jl.group_size(L, w.w_pretrained)
        assert G == step + 1
        check_decode(jl, kc, vc, qs[step], L, w.w0, w.w_pretrained, w.theta, f"decode L={L} G={G}")
        now = (kc.view(torch.int16).long().sum().item(), vc.view(torch.int16).long().sum().item())
        assert now == sums, "the KV cache was modified"


@pytest.mark.parametrize("L,Lcap,Hq,Hkv,wp,w0,d", [
    (1, 8, 4, 2, 4, 0, 128),          # only the new token
    (2, 2, 4, 4, 1, 0, 128),          # G = 2, w0 = 0
    (7, 40, 8, 1, 3, 2, 128),         # ragged, G = 3, 8 query heads per KV head
    (64, 64, 2, 2, 16, 5, 128),       # exactly one 64-key block
    (65, 100, 4, 1, 16, 0, 128),      # one key past a block
    (300, 300, 16, 8, 40, 17, 128),   # G = 8, local/remote boundary inside a warp step
    (1000, 1200, 32, 8, 300, 64, 128),
    (1000, 1000, 8, 8, 2000, 10, 128),  # G = 1
    (777, 800, 4, 2, 100, 776, 128),  # w0 >= L-1: all local at G = 8
    (500, 512, 4, 2, 100, 30, 64),    # d = 64
    (777, 800, 64, 8, 100, 20, 64),   # d = 64, 8 query heads per KV head
    (2000, 2000, 16, 16, 500, 300, 64),  # d = 64, 16 KV heads (two head groups), MHA
    (1000, 1000, 32, 16, 300, 64, 128),  # 16 KV heads (two head groups of 8)
    (129, 200, 9, 9, 40, 3, 128),     # 9 KV heads: head groups of 5 and 4
    (600, 650, 12, 4, 200, 50, 128),  # 3 query heads per KV head
    (800, 800, 40, 8, 250, 100, 128),  # 5 query heads per KV head (Qwen3-14B layout)
    (5000, 5000, 24, 4, 1000, 333, 64),  # 6 query heads per KV head, d = 64, G = 5
])
def test_decode_small(jl, L, Lcap, Hq, Hkv, wp, w0, d):
    kc, vc, qs = synth.decode_inputs(Lcap, Hq, Hkv, d, L + 3 * w0, 1)
    check_decode(jl, kc.cuda(), vc.cuda(), qs[0], L, w0, wp, 1e4, f"L={L} Hq={Hq} Hkv={Hkv} d={d}")


def test_decode_batch(jl):
    kc, vc, qs = synth.decode_inputs(500, 8, 2, 128, 9, 1, B=3)
    check_decode(jl, kc.cuda(), vc.cuda(), qs[0], 450, 30, 100, 1e6, "B=3")


@pytest.mark.parametrize("d", [128, 64])
def test_decode_matches_prefill_rows(jl, d):
    """Prefill fills the cache (k_rot_out); decode at length L' then agrees
    with prefill row L'-1 when both see the same G (here L' > w_p * (G-1))."""
    import torch
    L, Hq, Hkv, wp, w0 = 700, 8, 2, 200, 50
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, 21)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    krot = torch.empty_like(kd)
    o_pre, lse_pre = jl.prefill(qd, kd, vd, w0, wp, 1e4, k_rot_out=krot)
    for Lp in (601, 650, 700):  # G(Lp) == G(700) == 4
        o_dec, lse_dec = jl.decode(qd[:, Lp - 1].contiguous(), krot, vd, Lp, w0, wp, 1e4)
        assert np.abs(to_np(o_dec) - to_np(o_pre[:, Lp - 1])).max() <= 3e-2, Lp
        assert np.abs(to_np(lse_dec) - to_np(lse_pre[:, :, Lp - 1])).max() <= 2e-3, Lp
    jl.device_status()


@pytest.mark.parametrize("lengths,Hq,Hkv,wp,w0", [
    ((1, 300, 4097, 9000), 32, 8, 2048, 512),     # G = 1, 1, 3, 5 in one batch
    ((65, 64, 63, 2), 8, 2, 16, 5),                # around one 64-key block
    ((5000, 17), 4, 4, 6000, 100),                 # G = 1 everywhere
])
def test_decode_varlen(jl, lengths, Hq, Hkv, wp, w0):
    """Batched decode with per-sequence lengths: each sequence matches the
    oracle decode at its own length (its own G and query position)."""
    import torch
    B, Lcap = len(lengths), max(lengths) + 100
    kc, vc, qs = synth.decode_inputs(Lcap, Hq, Hkv, 128, sum(lengths), 1, B=B)
    kcd, vcd = kc.cuda(), vc.cuda()
    seq = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    o, lse = jl.decode_varlen(qs[0].cuda(), kcd, vcd, seq, w0, wp, 1e4)
    jl.device_status()
    for b, L in enumerate(lengths):
        o_ref, l_ref = oracle.bifocal_decode(qs[0][b:b + 1].float().numpy(), kc[b:b + 1, :L].float().numpy(),
                                             vc[b:b + 1, :L].float().numpy(), L, w0, wp, 1e4)
        assert_close(to_np(o[b:b + 1]), to_np(lse[b:b + 1]), o_ref, l_ref, f"sequence {b}, L={L}")


def test_decode_varlen_flags_bad_lengths(jl):
    """A length outside [1, Lcap] is clamped and reported by device_status."""
    import torch
    from bifocal_rope_extension_causal_b300 import JetLongError
    kc, vc, qs = synth.decode_inputs(200, 8, 2, 128, 3, 1, B=2)
    seq = torch.tensor([150, 999], dtype=torch.int32, device="cuda")
    jl.decode_varlen(qs[0].cuda(), kc.cuda(), vc.cuda(), seq, 10, 64, 1e4, max_len=200)
    with pytest.raises(JetLongError):
        jl.device_status()
    jl.device_status()  # cleared


def test_decode_in_cuda_graph(jl):
    """A decode step captured in a CUDA graph (the serving form: no host work
    per step) replays to the eager result."""
    import torch
    kc, vc, qs = synth.decode_inputs(3000, 8, 2, 128, 77, 1)
    kc, vc, q = kc.cuda(), vc.cuda(), qs[0].cuda()
    o_ref, l_ref = jl.decode(q, kc, vc, 2500, 100, 1000, 1e4)
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(l_ref)
    ws = jl.alloc_workspace(jl.decode_workspace_size(1, 8, 128, 3000), q.device)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        jl.decode(q, kc, vc, 2500, 100, 1000, 1e4, out=o, lse=lse, workspace=ws)
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        jl.decode(q, kc, vc, 2500, 100, 1000, 1e4, out=o, lse=lse, workspace=ws)
    o.zero_()
    lse.zero_()
    graph.replay()
    torch.cuda.synchronize()
    jl.device_status()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
