"""Failure detection without a GPU fault: a kernel waits, with the library's
bounded wait, on a barrier that nothing arrives on; the wait runs out, the
kernel records a status code and returns, and the host reads it through
jl_device_status.  The context stays usable afterwards."""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import bifocal_rope_extension_causal_b300 as jl
    from bifocal_rope_extension_causal_b300 import _capi, build, synth
    build.build()
    lib = _capi.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.jl_device_status(stream) == _capi.JL_OK
    _capi.check(lib.jl_selftest_bounded_wait(2_000_000, stream))  # ~1 ms
    assert lib.jl_device_status(stream) == _capi.JL_ERR_TIMEOUT
    assert b"bounded device wait" in lib.jl_last_error()
    assert lib.jl_device_status(stream) == _capi.JL_OK  # read-and-clear
    # The context is still usable: a prefill runs and is finite.
    q, k, v = synth.prefill_inputs(300, 4, 2, 128, 1)
    o, lse = jl.prefill(q.cuda(), k.cuda(), v.cuda(), 16, 100, 1e4)
    jl.device_status()
    assert np.isfinite(o.float().cpu().numpy()).all()


def test_selftest_argument_check():
    from bifocal_rope_extension_causal_b300 import _capi, build
    build.build()
    assert _capi.load().jl_selftest_bounded_wait(0, None) == _capi.JL_ERR_INVALID


@pytest.mark.parametrize("kernel", ["single_cta", "cta_pair"])
@pytest.mark.parametrize("limit", [1, 300])
def test_prefill_pipeline_timeout_is_reported_and_context_survives(limit, kernel):
    """The real attention pipeline with a wait limit small enough to run out:
    its CTAs give up, drain their bulk copies and tensor-core work, free
    their tensor memory and return; jl_device_status reports the timeout and
    a normal prefill on the same context then matches the oracle."""
    import torch
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import oracle
    import bifocal_rope_extension_causal_b300 as jl
    from bifocal_rope_extension_causal_b300 import _capi, build, synth
    from gpu_common import assert_close, to_np
    build.build()
    lib = _capi.load()
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    # G = 4 with a small window: remote visits, local visits, straddling
    # tiles and the mid-CTA reload of Q all occur.
    L, Hq, Hkv, d, wp, w0, theta = 512, 4, 2, 128, 128, 16, 1e4
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, 5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.zeros_like(qd)
    lse = torch.zeros((1, Hq, L), dtype=torch.float32, device="cuda")
    nbytes = jl.prefill_workspace_size(1, L, Hq, Hkv, d, wp)
    ws = jl.alloc_workspace(nbytes, qd.device)
    assert lib.jl_device_status(stream) == _capi.JL_OK
    selftest = (lib.jl_selftest_prefill_wait_limit if kernel == "single_cta"
                else lib.jl_selftest_prefill_pair_wait_limit)
    _capi.check(selftest(P(qd.data_ptr()), P(kd.data_ptr()), P(vd.data_ptr()), P(o.data_ptr()), P(lse.data_ptr()),
                         1, L, Hq, Hkv, d, w0, wp, theta, limit, P(ws.data_ptr()), nbytes, stream))
    assert lib.jl_device_status(stream) == _capi.JL_ERR_TIMEOUT
    assert b"bounded device wait" in lib.jl_last_error()
    assert lib.jl_device_status(stream) == _capi.JL_OK  # read-and-clear
    o2, l2 = jl.prefill(qd, kd, vd, w0, wp, theta, workspace=ws)
    if kernel == "cta_pair":  # the same kernel again, without the limit
        _capi.check(lib.jl_bifocal_attention_cta_pair(P(vd.data_ptr()), P(o2.data_ptr()), P(l2.data_ptr()), 1, L,
                                                      Hq, Hkv, d, w0, wp, 0.0, P(ws.data_ptr()), nbytes, stream))
    jl.device_status()
    o_ref, l_ref = oracle.bifocal_prefill(q.float().numpy(), k.float().numpy(), v.float().numpy(), w0, wp, theta,
                                          round_rotated_qk=True)
    assert_close(to_np(o2), to_np(l2), o_ref, l_ref, f"prefill after a timeout (limit {limit})")


def test_prefill_selftest_argument_check():
    from bifocal_rope_extension_causal_b300 import _capi, build
    build.build()
    lib = _capi.load()
    rc = lib.jl_selftest_prefill_wait_limit(1 << 20, 1 << 20, 1 << 20, 1 << 20, None, 1, 64, 2, 1, 128, 4, 16,
                                            1e4, 0, 1 << 20, 1 << 30, None)
    assert rc == _capi.JL_ERR_INVALID
    rc = lib.jl_selftest_prefill_pair_wait_limit(1 << 20, 1 << 20, 1 << 20, 1 << 20, None, 1, 64, 2, 1, 64, 4, 16,
                                                 1e4, 100, 1 << 20, 1 << 30, None)
    assert rc == _capi.JL_ERR_UNSUPPORTED
