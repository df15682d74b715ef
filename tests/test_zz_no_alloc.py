"""jl_bifocal_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (for example a plugin whose host framework owns every
device allocation and offers it no allocator).  It must give the same result
as jl_bifocal_decode with a caller workspace, call after call, although its
scratch lives in one fixed array shared by all calls.

This file is named so that pytest collects it last."""

import ctypes

import numpy as np
import pytest

from bifocal_rope_extension_causal_b300 import synth
from gpu_common import LSE_ABS, O_MAX_ABS

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_decode():
    import torch
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    from bifocal_rope_extension_causal_b300 import _capi, build
    build.build()
    lib = _capi.load()
    P = ctypes.c_void_p
    Lcap, Hq, Hkv, d, wp, w0, theta = 70000, 32, 8, 128, 32768, 4096, 1e6
    kc, vc, qs = synth.decode_inputs(Lcap, Hq, Hkv, d, 31, 2)
    kc, vc, qs = kc.cuda(), vc.cuda(), qs.cuda()
    stream = P(torch.cuda.current_stream().cuda_stream)
    ws_bytes = lib.jl_bifocal_decode_workspace_size(1, Hq, d, Lcap)
    assert 0 < ws_bytes <= lib.jl_bifocal_decode_noalloc_scratch_bytes()
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    # Two calls in a row with different lengths (G = 2 then 3): the second
    # must not see anything left in the shared scratch by the first.
    for step, L in enumerate((40000, 65537)):
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
        og, orf = o.float().cpu().numpy(), o_ref.float().cpu().numpy()
        lg, lrf = lse.cpu().numpy(), l_ref.cpu().numpy()
        assert np.isfinite(og).all() and np.isfinite(lg).all()
        assert np.abs(og - orf).max() <= O_MAX_ABS, step
        assert np.abs(lg - lrf).max() <= LSE_ABS, step


def test_noalloc_rejects_sizes_beyond_the_scratch():
    from bifocal_rope_extension_causal_b300 import _capi, build
    build.build()
    lib = _capi.load()
    # 64 query heads need more than the fixed array; rejected before any launch.
    rc = lib.jl_bifocal_decode_noalloc(1 << 20, 1 << 20, 1 << 20, 10, 16, 1 << 20, None, 1, 64, 8, 128,
                                       4, 8, 1e4, 0.0, None)
    assert rc == _capi.JL_ERR_UNSUPPORTED
    assert b"scratch" in lib.jl_last_error()
