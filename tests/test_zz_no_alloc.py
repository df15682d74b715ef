"""jl_bifocal_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (for example a plugin whose host framework owns every
device allocation and offers it no allocator).  It must give the same result
as jl_bifocal_decode with a caller workspace, call after call, although its
scratch lives in one fixed array shared by all calls.

This file is named so that pytest collects it last."""

import ctypes

import pytest

from bifocal_rope_extension_causal_b300 import synth

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_decode():
    import torch
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    from bifocal_rope_extension_causal_b300 import _capi, build
    build.build()
    lib = _capi.load()
    P = ctypes.c_void_p
    Lcap, Hq, Hkv, d, wp, w0, theta = 70000, 32, 8, 128, 32768, 4096, 1e6
    kc, vc, qs = synth.decode_inputs(Lcap, Hq, Hkv, d, 31, 3)
    kc, vc, qs = kc.cuda(), vc.cuda(), qs.cuda()
    stream = P(torch.cuda.current_stream().cuda_stream)
    ws_bytes = lib.jl_bifocal_decode_workspace_size(1, Hq, d, Lcap)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    # Calls in a row with different lengths and G (3, then 1 with far fewer
    # key slices, then 2): no call may see what an earlier, longer one left
    # in the shared scratch.  Same kernels and the same slicing as the
    # workspace decode, so the results must agree bit for bit.
    for step, L in enumerate((65537, 700, 40000)):
        q = qs[step]
        o_ref = torch.empty(1, Hq, d, dtype=torch.bfloat16, device="cuda")
        l_ref = torch.empty(1, Hq, dtype=torch.float32, device="cuda")
        _capi.check(lib.jl_bifocal_decode(P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()), L, Lcap,
                                          P(o_ref.data_ptr()), P(l_ref.data_ptr()), 1, Hq, Hkv, d, w0, wp,
                                          theta, 0.0, P(ws.data_ptr()), ws_bytes, stream))
        o = torch.full((1, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((1, Hq), float("nan"), dtype=torch.float32, device="cuda")
        _capi.check(lib.jl_bifocal_decode_noalloc(P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()), L,
                                                  Lcap, P(o.data_ptr()), P(lse.data_ptr()), 1, Hq, Hkv, d,
                                                  w0, wp, theta, 0.0, stream))
        _capi.check(lib.jl_device_status(stream))
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), step
        assert torch.equal(o, o_ref), (step, float((o.float() - o_ref.float()).abs().max()))
        assert torch.equal(lse, l_ref), (step, float((lse - l_ref).abs().max()))


def test_noalloc_rejects_sizes_beyond_the_scratch():
    from bifocal_rope_extension_causal_b300 import _capi, build
    build.build()
    lib = _capi.load()
    # 64 sequences x 512 query heads need more than the fixed array even at
    # one key slice per head (64 * 512 * 130 * 4 bytes > 16 MiB): rejected
    # before any launch, so the placeholder addresses are never touched.
    B, Hq, Hkv, d = 64, 512, 64, 128
    assert B * Hq * (d + 2) * 4 > lib.jl_bifocal_decode_noalloc_scratch_bytes()
    rc = lib.jl_bifocal_decode_noalloc(1 << 20, 1 << 20, 1 << 20, 10, 16, 1 << 20, None, B, Hq, Hkv, d,
                                       4, 8, 1e4, 0.0, None)
    assert rc == _capi.JL_ERR_UNSUPPORTED
    assert b"scratch" in lib.jl_last_error()
