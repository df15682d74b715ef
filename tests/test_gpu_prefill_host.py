"""Prefill from host buffers (jl_bifocal_prefill_host): the pipelined copies
and per-chunk launches give results bit-identical to one device-buffer
jl_bifocal_prefill call on the same data, for any chunking."""

import numpy as np
import pytest

from bifocal_rope_extension_causal_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jl():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bifocal_rope_extension_causal_b300 as mod
    from bifocal_rope_extension_causal_b300 import build
    build.build()
    return mod


@pytest.mark.parametrize("B,L,Hq,Hkv,d,wp,w0,n_chunks", [
    (1, 1000, 4, 2, 128, 300, 50, 3),    # G = 4, ragged last chunk
    (2, 777, 8, 2, 64, 200, 20, 2),      # two sequences, d = 64
    (1, 4096, 8, 8, 128, 8192, 100, 4),  # G = 1
    (1, 300, 2, 1, 128, 50, 299, 0),     # automatic chunking (one chunk), all local
    (1, 5000, 16, 2, 128, 1700, 700, 7),  # G = 3, band across chunk boundaries
])
def test_host_prefill_equals_device_prefill(jl, B, L, Hq, Hkv, d, wp, w0, n_chunks):
    import torch
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, seed=L + n_chunks, B=B)
    o_ref, l_ref = jl.prefill(q.cuda(), k.cuda(), v.cuda(), w0, wp, 1e4)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = jl.prefill_host(qh, kh, vh, w0, wp, 1e4, n_chunks=n_chunks)
    torch.cuda.synchronize()
    jl.device_status()
    assert torch.equal(o, o_ref.cpu()), "o differs from the device-buffer prefill"
    assert torch.equal(lse, l_ref.cpu()), "lse differs from the device-buffer prefill"


def test_host_prefill_without_lse_and_repeated(jl):
    """lse may be omitted; back-to-back calls reuse the copy streams and events."""
    import torch
    q, k, v = synth.prefill_inputs(2048, 4, 2, 128, seed=3)
    o_ref, _ = jl.prefill(q.cuda(), k.cuda(), v.cuda(), 64, 512, 1e6)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    outs = [jl.prefill_host(qh, kh, vh, 64, 512, 1e6, want_lse=False, n_chunks=5)[0] for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, o_ref.cpu())


def test_host_prefill_pageable_buffers(jl):
    """Pageable (not page-locked) host tensors: the copies serialise with the
    host thread, and the results are still those of the device prefill."""
    import torch
    q, k, v = synth.prefill_inputs(1500, 4, 2, 128, seed=8)
    o_ref, l_ref = jl.prefill(q.cuda(), k.cuda(), v.cuda(), 40, 400, 1e4)
    out = torch.empty(q.shape, dtype=torch.bfloat16)
    lse = torch.empty((1, 4, 1500), dtype=torch.float32)
    o, l = jl.prefill_host(q, k, v, 40, 400, 1e4, out=out, lse=lse, n_chunks=3)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref.cpu()) and torch.equal(l, l_ref.cpu())
