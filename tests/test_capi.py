"""The C-ABI library builds, loads, and exports every symbol include/jetlong.h
declares; host-side logic (group size, workspace sizes, argument checks that
fail before any CUDA call) behaves as documented.  CPU only: no compute call
reaches the device here."""

import ctypes
import os
import re

import pytest

import bifocal_rope_extension_causal_b300 as jl
from bifocal_rope_extension_causal_b300 import _capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "jetlong.h")


@pytest.fixture(scope="module")
def lib():
    from bifocal_rope_extension_causal_b300 import build
    build.build()
    return _capi.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jl_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("jl_group_size", "jl_bifocal_prefill", "jl_bifocal_decode", "jl_last_error"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _capi.SIGNATURES, f"binding lacks a signature for {name}"


def test_group_size_matches_brute_force(lib):
    def brute(L, w):
        if L == 0:
            return 1
        g = 1
        while (L - 1) // g >= w:
            g += 1
        return g
    for w in (1, 2, 3, 64, 32768):
        for L in list(range(0, 300)) + [w - 1, w, w + 1, 2 * w + 1, 4 * w, 4 * w + 1]:
            if L >= 0:
                assert lib.jl_group_size(L, w) == brute(L, w), (L, w)
    assert lib.jl_group_size(-1, 5) == -1
    assert lib.jl_group_size(5, 0) == -1
    assert [jl.group_size(L, 32768) for L in (32767, 32769, 65537, 131072)] == [1, 2, 3, 4]


def test_workspace_sizes(lib):
    # G == 1 needs only the absolute copies; G > 1 both; plus the rotation
    # tables (3 * 1024 rows of d/2 float4).
    tables = 3 * 1024 * 64 * 16
    one = jl.prefill_workspace_size(1, 1024, 4, 2, 128, 4096)
    two = jl.prefill_workspace_size(1, 1024, 4, 2, 128, 512)
    assert one == 1024 * (4 + 2) * 128 * 2 + tables
    assert two == 2 * (one - tables) + tables
    three = lib.jl_bifocal_prefill_three_pass_workspace_size(1, 1024, 4, 2, 128, 512)
    assert three == two + 2 * 1024 * 4 * 128 * 2 + 3 * 4 * 1024 * 4
    assert jl.prefill_workspace_size(0, 1, 1, 1, 64, 1) == 0
    assert jl.decode_workspace_size(1, 32, 128, 131072) > 0
    assert jl.decode_workspace_size(1, 0, 128, 1) == 0


def _prefill_args(**kw):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, o=1 << 20, lse=None, B=1, L=128, Hq=2, Hkv=1, d=128,
             w0=16, wp=64, theta=1e4, scale=0.0, krot=None, ws=1 << 20, wsb=1 << 30, stream=None)
    a.update(kw)
    return (a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["L"], a["Hq"], a["Hkv"], a["d"],
            a["w0"], a["wp"], a["theta"], a["scale"], a["krot"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), _capi.JL_ERR_INVALID),
    (dict(L=0), _capi.JL_ERR_INVALID),
    (dict(Hq=3, Hkv=2), _capi.JL_ERR_INVALID),
    (dict(w0=-1), _capi.JL_ERR_INVALID),
    (dict(wp=0), _capi.JL_ERR_INVALID),
    (dict(theta=0.0), _capi.JL_ERR_INVALID),
    (dict(d=96), _capi.JL_ERR_UNSUPPORTED),
    (dict(q=(1 << 20) + 2), _capi.JL_ERR_INVALID),
    (dict(ws=None), _capi.JL_ERR_WORKSPACE),
    (dict(wsb=16), _capi.JL_ERR_WORKSPACE),
])
def test_prefill_argument_checks(lib, kw, code):
    """Rejected before any CUDA call: nothing is launched, the message says why."""
    assert lib.jl_bifocal_prefill(*_prefill_args(**kw)) == code
    assert lib.jl_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), _capi.JL_ERR_UNSUPPORTED),
    (dict(v=None), _capi.JL_ERR_INVALID),
    (dict(Hq=3, Hkv=2), _capi.JL_ERR_INVALID),
    (dict(wsb=16), _capi.JL_ERR_WORKSPACE),
])
def test_cta_pair_attention_argument_checks(lib, kw, code):
    """The CTA-pair kernel takes head dim 128 only and the attention checks."""
    a = dict(v=1 << 20, o=1 << 20, lse=None, B=1, L=128, Hq=2, Hkv=1, d=128, w0=16, wp=64, scale=0.0,
             ws=1 << 20, wsb=1 << 30, stream=None)
    a.update(kw)
    assert lib.jl_bifocal_attention_cta_pair(a["v"], a["o"], a["lse"], a["B"], a["L"], a["Hq"], a["Hkv"], a["d"],
                                             a["w0"], a["wp"], a["scale"], a["ws"], a["wsb"], a["stream"]) == code
    assert lib.jl_last_error().decode()


def _three_pass_args(**kw):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, o=1 << 20, lse=None, B=1, L=128, Hq=2, Hkv=1, d=128,
             w0=16, wp=64, theta=1e4, scale=0.0, ws=1 << 20, wsb=1 << 30, stream=None)
    a.update(kw)
    return (a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["L"], a["Hq"], a["Hkv"], a["d"],
            a["w0"], a["wp"], a["theta"], a["scale"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(v=None), _capi.JL_ERR_INVALID),
    (dict(Hq=3, Hkv=2), _capi.JL_ERR_INVALID),
    (dict(d=96), _capi.JL_ERR_UNSUPPORTED),
    (dict(L=1 << 30), _capi.JL_ERR_UNSUPPORTED),
    (dict(wsb=1 << 20), _capi.JL_ERR_WORKSPACE),
])
def test_three_pass_argument_checks(lib, kw, code):
    assert lib.jl_bifocal_prefill_three_pass(*_three_pass_args(**kw)) == code
    assert lib.jl_last_error().decode()


def _host_args(**kw):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, o=1 << 20, lse=None, B=1, L=128, Hq=2, Hkv=1, d=128,
             w0=16, wp=64, theta=1e4, scale=0.0, nc=0, ws=1 << 20, wsb=1 << 30, stream=None)
    a.update(kw)
    return (a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["L"], a["Hq"], a["Hkv"], a["d"],
            a["w0"], a["wp"], a["theta"], a["scale"], a["nc"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(o=None), _capi.JL_ERR_INVALID),
    (dict(nc=-1), _capi.JL_ERR_INVALID),
    (dict(theta=-1.0), _capi.JL_ERR_INVALID),
    (dict(B=0), _capi.JL_ERR_INVALID),
    (dict(d=32), _capi.JL_ERR_UNSUPPORTED),
    (dict(ws=None), _capi.JL_ERR_WORKSPACE),
    (dict(wsb=4096), _capi.JL_ERR_WORKSPACE),
])
def test_host_prefill_argument_checks(lib, kw, code):
    """Rejected before any CUDA call (host pointers are never dereferenced here)."""
    assert lib.jl_bifocal_prefill_host(*_host_args(**kw)) == code
    assert lib.jl_last_error().decode()


def test_host_prefill_workspace_size(lib):
    base = lib.jl_bifocal_prefill_workspace_size(2, 1000, 4, 2, 128, 300)
    host = lib.jl_bifocal_prefill_host_workspace_size(2, 1000, 4, 2, 128, 300)
    def up(x):
        return (x + 255) // 256 * 256
    assert host == base + 2 * up(2 * 1000 * 4 * 128 * 2) + 2 * up(2 * 1000 * 2 * 128 * 2) + up(2 * 4 * 1000 * 4)
    assert lib.jl_bifocal_prefill_host_workspace_size(0, 1000, 4, 2, 128, 300) == 0


def _decode_args(**kw):
    a = dict(q=1 << 20, kc=1 << 20, vc=1 << 20, L=10, Lcap=16, o=1 << 20, lse=None, B=1, Hq=4,
             Hkv=2, d=128, w0=4, wp=8, theta=1e4, scale=0.0, ws=1 << 20, wsb=1 << 30, stream=None)
    a.update(kw)
    return (a["q"], a["kc"], a["vc"], a["L"], a["Lcap"], a["o"], a["lse"], a["B"], a["Hq"],
            a["Hkv"], a["d"], a["w0"], a["wp"], a["theta"], a["scale"], a["ws"], a["wsb"],
            a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(kc=None), _capi.JL_ERR_INVALID),
    (dict(L=0), _capi.JL_ERR_INVALID),
    (dict(L=17), _capi.JL_ERR_INVALID),
    (dict(Hq=6, Hkv=4), _capi.JL_ERR_INVALID),
    (dict(d=96), _capi.JL_ERR_UNSUPPORTED),
    (dict(Hq=48, Hkv=3), _capi.JL_ERR_UNSUPPORTED),
    (dict(Hq=64, Hkv=4), _capi.JL_ERR_UNSUPPORTED),
    (dict(ws=None), _capi.JL_ERR_WORKSPACE),
])
def test_decode_argument_checks(lib, kw, code):
    assert lib.jl_bifocal_decode(*_decode_args(**kw)) == code
    assert lib.jl_last_error().decode()


@pytest.mark.parametrize("kw", [
    dict(kc=None), dict(L=0), dict(L=17), dict(Hq=6, Hkv=4), dict(d=96), dict(Hq=48, Hkv=3),
    dict(Hq=64, Hkv=4), dict(o=None, Hq=4096, Hkv=8), dict(Hkv=0, Hq=4096), dict(theta=0.0, Hq=4096),
])
def test_noalloc_decode_argument_checks_match_decode(lib, kw):
    """The allocation-free decode rejects bad arguments with the same codes as
    the workspace decode, before its scratch-size limit (the Hq = 4096 cases
    would also exceed the fixed scratch array)."""
    args = _decode_args(**kw)
    want = lib.jl_bifocal_decode(*args)
    assert want in (_capi.JL_ERR_INVALID, _capi.JL_ERR_UNSUPPORTED)
    got = lib.jl_bifocal_decode_noalloc(*args[:15], args[17])
    assert got == want, (kw, got, want)
    assert lib.jl_last_error().decode()


def test_decode_wider_shapes_pass_the_checks(lib):
    """d = 64, 16 KV heads and 3, 5, 6 query heads per KV head reach the
    workspace check (a small workspace is refused there, not the shape)."""
    for kw in (dict(d=64), dict(Hq=32, Hkv=16), dict(Hq=3, Hkv=1), dict(Hq=40, Hkv=8), dict(Hq=12, Hkv=2)):
        assert lib.jl_bifocal_decode(*_decode_args(wsb=16, **kw)) == _capi.JL_ERR_WORKSPACE, kw


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        jl.prefill(x, x[:, :, :1], x[:, :, :1], 4, 8, 1e4)


def test_product_path_does_not_import_the_oracle():
    """The package and its sources never reference the oracle."""
    pkg = os.path.join(ROOT, "bifocal_rope_extension_causal_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
