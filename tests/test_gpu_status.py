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
