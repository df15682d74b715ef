"""The three-pass inclusion-exclusion prefill (digest page, "Method", Eq. 7)
through the C ABI against the fp64 oracle, and against the routed single
pass on the same inputs.

Both forms compute the same function; the three-pass merge subtracts the
aliased window's mass (pass C) from the full aliased pass (B), so its error
is largest where the local window holds most of the attention.  The
fidelity printed by the A/B test (run with -s) is the evidence for the
comparison of the two forms."""

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


def both_forms(jl, q, k, v, w0, wp, theta):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = jl.prefill(qd, kd, vd, w0, wp, theta)
    o3, l3 = jl.prefill_three_pass(qd, kd, vd, w0, wp, theta)
    jl.device_status()
    return (to_np(o1), to_np(l1)), (to_np(o3), to_np(l3))


def errors(o, l, o_ref, l_ref):
    e = np.abs(o - o_ref)
    return float(e.max()), float(e.mean()), float(np.abs(l - l_ref).max())


@pytest.mark.parametrize("L,Hq,Hkv,d,wp,w0", [
    (1, 2, 1, 64, 64, 16),        # one row
    (63, 4, 2, 64, 16, 5),        # ragged tail, G = 4
    (129, 8, 2, 128, 40, 7),      # G = 4, three tiles
    (200, 4, 4, 64, 256, 16),     # G = 1: B = full causal, A = C
    (300, 2, 1, 128, 50, 299),    # w0 >= L - 1: A is everything, B - C = 0
    (333, 6, 2, 128, 37, 100),    # G = 10, band across several tiles
    (2304, 8, 8, 128, 300, 400),  # G = 8, many tiles
])
def test_three_pass_matches_oracle(jl, L, Hq, Hkv, d, wp, w0):
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, seed=L + 5 * w0)
    _, (o3, l3) = both_forms(jl, q, k, v, w0, wp, 1e4)
    qn, kn, vn = (x.float().numpy() for x in (q, k, v))
    o_r, l_r = oracle.bifocal_prefill(qn, kn, vn, w0, wp, 1e4, round_rotated_qk=True)
    o_p, _ = oracle.bifocal_prefill(qn, kn, vn, w0, wp, 1e4)
    tag = f"three-pass L={L} Hq={Hq} Hkv={Hkv} d={d} wp={wp} w0={w0}"
    assert_close(o3, l3, o_r, l_r, tag + " (rounded oracle)")
    err = np.abs(o3 - o_p)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, tag + " (plain oracle)"


def test_three_pass_equals_single_pass_mid(jl):
    """The two forms agree on a mid-size case (G = 3, GQA 8, band over many tiles)."""
    q, k, v = synth.prefill_inputs(5000, 16, 2, 128, seed=9)
    (o1, l1), (o3, l3) = both_forms(jl, q, k, v, 700, 1700, 1e6)
    assert np.abs(o1 - o3).max() <= 2e-2 and np.abs(o1 - o3).mean() <= 2e-3
    assert np.abs(l1 - l3).max() <= 1e-3


def peaked_local_inputs(L, Hq, Hkv, d, seed, gain):
    """Queries equal to their own (scaled) keys: the diagonal and its
    neighbourhood dominate, so most of B's mass lies in the window that C
    removes again -- the cancelling case of the inclusion-exclusion merge."""
    import torch
    q, k, v = synth.prefill_inputs(L, Hq, Hkv, d, seed)
    rep = Hq // Hkv
    kk = k.float().repeat_interleave(rep, dim=2)
    q = (gain * kk + 0.3 * q.float()).to(torch.bfloat16)
    return q, k, v


# The three-pass merge combines three bf16-rounded outputs; where the window
# dominates, w_A ~ w_B ~ w_C and den ~ w_A, so its O error is about three
# times one pass's output rounding (2.7e-2 measured, against the 2e-2
# acceptance bound that the routed single pass meets).  The A/B form is held
# to twice the acceptance bound in that case, and the public header states
# the measured figure: this is a documented limit of the A/B entry point,
# not the acceptance bound of the prefill.
THREE_PASS_CANCEL_O_MAX = 4e-2


@pytest.mark.parametrize("gain", [1.0, 2.0])
def test_fidelity_ab_peaked_local(jl, gain):
    """A/B of the two forms on a case where the local window dominates (the
    cancelling case of the merge).  The printed errors compare them."""
    L, Hq, Hkv, d, wp, w0 = 1024, 4, 2, 128, 256, 64
    q, k, v = peaked_local_inputs(L, Hq, Hkv, d, 31, gain)
    (o1, l1), (o3, l3) = both_forms(jl, q, k, v, w0, wp, 1e4)
    qn, kn, vn = (x.float().numpy() for x in (q, k, v))
    o_r, l_r = oracle.bifocal_prefill(qn, kn, vn, w0, wp, 1e4, round_rotated_qk=True)
    e1, e3 = errors(o1, l1, o_r, l_r), errors(o3, l3, o_r, l_r)
    print(f"\npeaked-local gain={gain}: single pass O max/mean {e1[0]:.3e}/{e1[1]:.3e} LSE {e1[2]:.3e}; "
          f"three-pass O max/mean {e3[0]:.3e}/{e3[1]:.3e} LSE {e3[2]:.3e}")
    assert_close(o1, l1, o_r, l_r, f"single pass, peaked local gain={gain}")
    assert np.isfinite(o3).all() and np.isfinite(l3).all()
    assert e3[0] <= THREE_PASS_CANCEL_O_MAX and e3[1] <= 2e-3 and e3[2] <= 1e-3, e3


def test_three_pass_64k_sampled_rows(jl):
    """The 2x-extension workload (L = 65536, G = 2) on 512 seeded rows per head."""
    w = W.EXT_64K
    q, k, v = synth.prefill_inputs(w.L, w.Hq, w.Hkv, w.d, w.index)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = jl.prefill_three_pass(qd, kd, vd, w.w0, w.w_pretrained, w.theta)
    jl.device_status()
    G = jl.group_size(w.L, w.w_pretrained)
    rows = np.stack([sample_rows(w.L, w.w0, w.w_pretrained, G, 512, 1000 * w.index + h)
                     for h in range(w.Hq)])
    og = np.stack([to_np(o[0, rows[h], h]) for h in range(w.Hq)], axis=1)[None]
    lg = np.stack([to_np(lse[0, h, rows[h]]) for h in range(w.Hq)])[None]
    del o, lse, qd, kd, vd
    qn, kn, vn = (x.float().numpy() for x in (q, k, v))
    o_r, l_r = oracle_prefill_rows(qn, kn, vn, w.w0, w.w_pretrained, w.theta, rows, True)
    e = assert_close(og, lg, o_r, l_r, "three-pass " + w.name)
    print(f"\nthree-pass {w.name}: O max/mean {e[0]:.3e}/{e[1]:.3e} LSE {e[2]:.3e}")
