"""Causal bifocal-RoPE attention (dynamic bifocal RoPE, "Jet-Long") on B300.

Thin Python layer over libjetlong.so (include/jetlong.h): the functions
below check tensor placement and layout, allocate outputs and workspace with
torch, and call the C ABI on the current CUDA stream.  All arithmetic runs
in the library's sm_103a kernels.
"""

from __future__ import annotations

import ctypes

from . import _capi
from ._capi import JetLongError, check, load  # noqa: F401

__all__ = [
    "group_size",
    "prefill_workspace_size",
    "decode_workspace_size",
    "prefill",
    "prefill_chunk",
    "prefill_three_pass",
    "prefill_host",
    "decode",
    "decode_varlen",
    "device_status",
    "JetLongError",
]


def _torch():
    import torch
    return torch


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda_bf16(name, t, ndim):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor, got shape {tuple(t.shape)}")


def group_size(L: int, w_pretrained: int) -> int:
    """G = max(1, ceil(L / w_pretrained)) from the library (-1 for bad args)."""
    return int(load().jl_group_size(int(L), int(w_pretrained)))


def prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained) -> int:
    return int(load().jl_bifocal_prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained))


def decode_workspace_size(B, Hq, d, Lcap) -> int:
    return int(load().jl_bifocal_decode_workspace_size(B, Hq, d, Lcap))


def alloc_workspace(nbytes: int, device):
    """A 256-byte-aligned uint8 device buffer (torch's allocator aligns to 512)."""
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def prefill(q, k, v, w0: int, w_pretrained: int, rope_theta: float, softmax_scale: float = 0.0,
            *, out=None, lse=None, want_lse: bool = True, k_rot_out=None, workspace=None,
            stream=None):
    """Causal bifocal-RoPE prefill.  q [B, L, Hq, d], k/v [B, L, Hkv, d] bf16
    CUDA tensors (raw, pre-RoPE).  Returns (o [B, L, Hq, d] bf16,
    lse [B, Hq, L] fp32 or None)."""
    torch = _torch()
    _need_cuda_bf16("q", q, 4)
    _need_cuda_bf16("k", k, 4)
    _need_cuda_bf16("v", v, 4)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device)
    nbytes = prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained)
    if workspace is None:
        workspace = alloc_workspace(nbytes, q.device)
    check(load().jl_bifocal_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, Hq, Hkv, d, int(w0),
        int(w_pretrained), float(rope_theta), float(softmax_scale), _ptr(k_rot_out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, lse


def prefill_three_pass(q, k, v, w0: int, w_pretrained: int, rope_theta: float, softmax_scale: float = 0.0,
                       *, out=None, lse=None, want_lse: bool = True, workspace=None, stream=None):
    """The same prefill in its three-pass inclusion-exclusion form (two window
    passes and one full aliased pass, merged).  Same arguments and outputs as
    prefill (no k_rot_out)."""
    torch = _torch()
    _need_cuda_bf16("q", q, 4)
    _need_cuda_bf16("k", k, 4)
    _need_cuda_bf16("v", v, 4)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(load().jl_bifocal_prefill_three_pass_workspace_size(
            B, L, Hq, Hkv, d, int(w_pretrained)), q.device)
    check(load().jl_bifocal_prefill_three_pass(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, Hq, Hkv, d, int(w0),
        int(w_pretrained), float(rope_theta), float(softmax_scale),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, lse


def _need_host_bf16(name, t, ndim):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a CPU tensor (page-locked for overlapped copies)")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor, got shape {tuple(t.shape)}")


def prefill_host(q, k, v, w0: int, w_pretrained: int, rope_theta: float, softmax_scale: float = 0.0,
                 *, out=None, lse=None, want_lse: bool = True, n_chunks: int = 0, workspace=None,
                 device=None, stream=None):
    """Prefill from host buffers: q [B, L, Hq, d], k/v [B, L, Hkv, d] bf16 CPU
    tensors (pinned for overlap).  The library copies chunks in, computes and
    copies o [B, L, Hq, d] and lse [B, Hq, L] back into host tensors (pinned,
    allocated if not given).  The outputs are complete after the stream
    synchronises.  Returns (o, lse)."""
    torch = _torch()
    _need_host_bf16("q", q, 4)
    _need_host_bf16("k", k, 4)
    _need_host_bf16("v", v, 4)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, L), dtype=torch.float32).pin_memory()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if workspace is None:
        workspace = alloc_workspace(load().jl_bifocal_prefill_host_workspace_size(
            B, L, Hq, Hkv, d, int(w_pretrained)), dev)
    check(load().jl_bifocal_prefill_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, Hq, Hkv, d, int(w0), int(w_pretrained),
        float(rope_theta), float(softmax_scale), int(n_chunks), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, lse


def prefill_chunk(q, k, v, k_cache, v_cache, P0: int, w0: int, w_pretrained: int,
                  rope_theta: float, softmax_scale: float = 0.0, *, out=None, lse=None,
                  want_lse: bool = True, workspace=None, stream=None):
    """Chunked prefill: q [B, C, Hq, d], k/v [B, C, Hkv, d] raw chunk tokens at
    positions P0 .. P0+C-1; k_cache/v_cache [B, Lcap, Hkv, d] hold positions
    0 .. P0-1 and receive the chunk.  Returns (o [B, C, Hq, d], lse [B, Hq, C])."""
    torch = _torch()
    for name, t, nd in (("q", q, 4), ("k", k, 4), ("v", v, 4), ("k_cache", k_cache, 4),
                        ("v_cache", v_cache, 4)):
        _need_cuda_bf16(name, t, nd)
    B, C, Hq, d = q.shape
    Hkv, Lcap = k.shape[2], k_cache.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, C), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(load().jl_bifocal_prefill_chunk_workspace_size(
            B, C, int(P0), Hq, Hkv, d, int(w_pretrained)), q.device)
    check(load().jl_bifocal_prefill_chunk(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), int(P0), Lcap, _ptr(out), _ptr(lse),
        B, C, Hq, Hkv, d, int(w0), int(w_pretrained), float(rope_theta), float(softmax_scale),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, lse


def decode(q, k_cache, v_cache, L: int, w0: int, w_pretrained: int, rope_theta: float,
           softmax_scale: float = 0.0, *, out=None, lse=None, want_lse: bool = True,
           workspace=None, stream=None):
    """One decode step.  q [B, Hq, d] raw; k_cache/v_cache [B, Lcap, Hkv, d]
    bf16 CUDA tensors (keys rotated at their absolute positions).  Returns
    (o [B, Hq, d] bf16, lse [B, Hq] fp32 or None)."""
    torch = _torch()
    _need_cuda_bf16("q", q, 3)
    _need_cuda_bf16("k_cache", k_cache, 4)
    _need_cuda_bf16("v_cache", v_cache, 4)
    B, Hq, d = q.shape
    Lcap, Hkv = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(decode_workspace_size(B, Hq, d, Lcap), q.device)
    check(load().jl_bifocal_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), int(L), Lcap, _ptr(out), _ptr(lse), B, Hq, Hkv, d,
        int(w0), int(w_pretrained), float(rope_theta), float(softmax_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, lse


def decode_varlen(q, k_cache, v_cache, seqlens, w0: int, w_pretrained: int, rope_theta: float,
                  softmax_scale: float = 0.0, *, max_len=None, out=None, lse=None, want_lse: bool = True,
                  workspace=None, stream=None):
    """Batched decode, one length per sequence.  seqlens: int32 CUDA tensor [B]
    (sequence b's new token is at position seqlens[b] - 1).  Returns
    (o [B, Hq, d], lse [B, Hq])."""
    torch = _torch()
    _need_cuda_bf16("q", q, 3)
    _need_cuda_bf16("k_cache", k_cache, 4)
    _need_cuda_bf16("v_cache", v_cache, 4)
    if not (isinstance(seqlens, torch.Tensor) and seqlens.is_cuda and seqlens.dtype == torch.int32
            and seqlens.dim() == 1 and seqlens.is_contiguous()):
        raise TypeError("seqlens must be a contiguous 1-d int32 CUDA tensor")
    B, Hq, d = q.shape
    Lcap, Hkv = k_cache.shape[1], k_cache.shape[2]
    if max_len is None:
        max_len = int(seqlens.max().item())
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(decode_workspace_size(B, Hq, d, Lcap), q.device)
    check(load().jl_bifocal_decode_varlen(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), int(max_len), Lcap, _ptr(out), _ptr(lse), B, Hq,
        Hkv, d, int(w0), int(w_pretrained), float(rope_theta), float(softmax_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))
    return out, lse


def device_status(stream=None) -> None:
    """Sync the stream and raise JetLongError if a bounded device wait ran out."""
    check(load().jl_device_status(_stream_ptr(stream)))
