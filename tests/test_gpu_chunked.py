"""Chunked prefill against an absolute-position cache.  Each chunk is checked
against the oracle's chunked prefill fed the cache exactly as the GPU stored
it (bf16 R_k x_k; remote cached keys take the correction rotation of the
stored key, as in the digest page's "KV cache invariant"), O also against
the full-prefill rows; the cache receives R_k x_k and v, and earlier cache
rows are never modified."""

import numpy as np
import pytest

import oracle
from bifocal_rope_extension_causal_b300 import synth
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


@pytest.mark.parametrize("L,Hq,Hkv,d,wp,w0,chunks", [
    (700, 8, 2, 128, 200, 50, (200, 250, 250)),       # G = 1 -> 3 -> 4 across chunks
    (1000, 4, 1, 128, 300, 0, (1, 299, 300, 400)),    # a one-token chunk, w0 = 0
    (513, 4, 2, 64, 128, 64, (256, 257)),             # d = 64, ragged
    (900, 4, 4, 128, 2000, 100, (450, 450)),          # G = 1 throughout
])
def test_chunks_equal_full_prefill_rows(jl, L, Hq, Hkv, d, wp, w0, chunks):
    import torch
    assert sum(chunks) == L
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, L + w0)
    kc = torch.zeros(1, L + 64, Hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    qn, kn, vn = (x.float().numpy() for x in (q, k, v))
    P0 = 0
    for C in chunks:
        before = kc[:, :P0].clone()
        o, lse = jl.prefill_chunk(q[:, P0:P0 + C].cuda(), k[:, P0:P0 + C].cuda(), v[:, P0:P0 + C].cuda(),
                                  kc, vc, P0, w0, wp, 1e4)
        jl.device_status()
        assert torch.equal(kc[:, :P0], before), "cached rows were modified"
        Lt = P0 + C
        o_r, l_r = oracle.bifocal_prefill_chunk(qn[:, P0:Lt], kn[:, P0:Lt], vn, to_np(before), P0, w0, wp,
                                                1e4, round_rotated_qk=True)
        assert_close(to_np(o), to_np(lse), o_r, l_r, f"chunk [{P0}, {Lt})")
        o_f, _ = oracle.bifocal_prefill(qn[:, :Lt], kn[:, :Lt], vn[:, :Lt], w0, wp, 1e4,
                                        round_rotated_qk=True, rows=np.arange(P0, Lt))
        err = np.abs(to_np(o) - o_f)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, f"chunk [{P0}, {Lt}) vs full prefill"
        P0 = Lt
    # The cache now holds R_k x_k (bf16) and v.
    ref = oracle.rope_rotate(kn[0], np.arange(L), 1e4)
    got = to_np(kc)[0, :L]
    assert np.abs(got - ref).max() <= 2.0 ** -8 * max(1.0, np.abs(ref).max())
    assert torch.equal(vc[:, :L].cpu(), v)


def test_chunked_cache_feeds_decode(jl):
    """Prefill in two chunks, then decode the next token from the filled cache."""
    import torch
    L, Hq, Hkv, d, wp, w0 = 600, 8, 2, 128, 150, 40
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, 77)
    kc = torch.zeros(1, L, Hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    jl.prefill_chunk(q[:, :300].cuda(), k[:, :300].cuda(), v[:, :300].cuda(), kc, vc, 0, w0, wp, 1e4)
    o2, lse2 = jl.prefill_chunk(q[:, 300:].cuda(), k[:, 300:].cuda(), v[:, 300:].cuda(), kc, vc, 300, w0,
                                wp, 1e4)
    od, ld = jl.decode(q[:, L - 1].cuda().contiguous(), kc, vc, L, w0, wp, 1e4)
    jl.device_status()
    assert np.abs(to_np(od) - to_np(o2[:, -1])).max() <= 3e-2
    assert np.abs(to_np(ld) - to_np(lse2[:, :, -1])).max() <= 2e-3


def test_chunk_argument_checks(jl):
    from bifocal_rope_extension_causal_b300 import _capi
    lib = _capi.load()
    P = 1 << 20
    # P0 + C > Lcap
    rc = lib.jl_bifocal_prefill_chunk(P, P, P, P, P, 10, 12, P, None, 1, 5, 2, 1, 128, 4, 8, 1e4, 0.0,
                                      P, 1 << 30, None)
    assert rc == _capi.JL_ERR_INVALID
