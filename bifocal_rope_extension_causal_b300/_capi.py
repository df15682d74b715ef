"""ctypes binding of libjetlong.so (include/jetlong.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  torch is used for device memory and streams; the
functions take CUDA tensors and pass their data pointers.  There is no CPU
fallback: a missing library or a non-CUDA tensor raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libjetlong.so")

JL_OK = 0
JL_ERR_INVALID = -1
JL_ERR_UNSUPPORTED = -2
JL_ERR_CUDA = -3
JL_ERR_TIMEOUT = -4
JL_ERR_WORKSPACE = -5

# Every symbol include/jetlong.h declares, with (restype, argtypes).
_c = ctypes
SIGNATURES = {
    "jl_group_size": (_c.c_int64, [_c.c_int64, _c.c_int64]),
    "jl_bifocal_prefill_workspace_size": (_c.c_size_t, [_c.c_int] * 6),
    "jl_bifocal_prefill": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k, v
        _c.c_void_p, _c.c_void_p,                          # o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, L, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double,                   # w0, w_pretrained, theta
        _c.c_float, _c.c_void_p,                           # softmax_scale, k_rot_out
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_rope": (_c.c_int, [
        _c.c_void_p, _c.c_void_p,                          # q, k
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, L, Hq, Hkv, d
        _c.c_int, _c.c_double, _c.c_void_p,                # w_pretrained, theta, k_rot_out
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_attention": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # v, o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, L, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_float,                    # w0, w_pretrained, softmax_scale
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_attention_cta_pair": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # v, o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, L, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_float,                    # w0, w_pretrained, softmax_scale
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_prefill_chunk_workspace_size": (_c.c_size_t, [_c.c_int] * 7),
    "jl_bifocal_prefill_chunk": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k, v (chunk, raw)
        _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_int,      # k_cache, v_cache, P0, Lcap
        _c.c_void_p, _c.c_void_p,                          # o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, C, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double, _c.c_float,       # w0, w_pretrained, theta, scale
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_prefill_three_pass_workspace_size": (_c.c_size_t, [_c.c_int] * 6),
    "jl_bifocal_prefill_three_pass": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k, v
        _c.c_void_p, _c.c_void_p,                          # o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, L, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double, _c.c_float,       # w0, w_pretrained, theta, scale
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_prefill_host_workspace_size": (_c.c_size_t, [_c.c_int] * 6),
    "jl_bifocal_prefill_host": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k, v (host)
        _c.c_void_p, _c.c_void_p,                          # o, lse (host)
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, L, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double, _c.c_float,       # w0, w_pretrained, theta, scale
        _c.c_int,                                          # n_chunks
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_decode_workspace_size": (_c.c_size_t, [_c.c_int] * 4),
    "jl_bifocal_decode": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k_cache, v_cache
        _c.c_int, _c.c_int, _c.c_void_p, _c.c_void_p,      # L, Lcap, o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int,            # B, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double, _c.c_float,       # w0, w_pretrained, theta, scale
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_decode_varlen": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k_cache, v_cache
        _c.c_void_p, _c.c_int, _c.c_int,                   # seqlens (device), max_len, Lcap
        _c.c_void_p, _c.c_void_p,                          # o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int,            # B, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double, _c.c_float,       # w0, w_pretrained, theta, scale
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_bifocal_decode_noalloc": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k_cache, v_cache
        _c.c_int, _c.c_int, _c.c_void_p, _c.c_void_p,      # L, Lcap, o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int,            # B, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double, _c.c_float,       # w0, w_pretrained, theta, scale
        _c.c_void_p,                                       # stream
    ]),
    "jl_bifocal_decode_noalloc_scratch_bytes": (_c.c_size_t, []),
    "jl_device_status": (_c.c_int, [_c.c_void_p]),
    "jl_selftest_bounded_wait": (_c.c_int, [_c.c_longlong, _c.c_void_p]),
    "jl_selftest_prefill_wait_limit": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k, v
        _c.c_void_p, _c.c_void_p,                          # o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, L, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double,                   # w0, w_pretrained, theta
        _c.c_longlong,                                     # limit_cycles
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_selftest_prefill_pair_wait_limit": (_c.c_int, [
        _c.c_void_p, _c.c_void_p, _c.c_void_p,            # q, k, v
        _c.c_void_p, _c.c_void_p,                          # o, lse
        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,  # B, L, Hq, Hkv, d
        _c.c_int, _c.c_int, _c.c_double,                   # w0, w_pretrained, theta
        _c.c_longlong,                                     # limit_cycles
        _c.c_void_p, _c.c_size_t, _c.c_void_p,             # workspace, bytes, stream
    ]),
    "jl_last_error": (_c.c_char_p, []),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libjetlong.so and declare every exported signature."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -m bifocal_rope_extension_causal_b300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


class JetLongError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def check(code: int) -> None:
    if code != JL_OK:
        raise JetLongError(code, load().jl_last_error().decode(errors="replace"))
