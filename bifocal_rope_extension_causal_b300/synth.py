"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the attention method: it only draws
standard-normal tensors from a seeded CPU generator and rounds them to bf16
(round to nearest even), so that both sides see identical bits.

Recipe (one generator per workload, seeded with the workload's index):
  prefill:  q [B, L, Hq, d], then k [B, L, Hkv, d], then v [B, L, Hkv, d]
  decode:   k_cache [B, Lcap, Hkv, d] (read as keys already rotated at their
            absolute position), then v_cache, then one raw query [B, Hq, d]
            per decode step.
"""

from __future__ import annotations

import torch


def _draw(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(L: int, Hq: int, Hkv: int, d: int, seed: int, B: int = 1):
    """(q, k, v) bf16 CPU tensors: q [B, L, Hq, d]; k, v [B, L, Hkv, d]."""
    g = torch.Generator().manual_seed(int(seed))
    q = _draw((B, L, Hq, d), g)
    k = _draw((B, L, Hkv, d), g)
    v = _draw((B, L, Hkv, d), g)
    return q, k, v


def decode_inputs(Lcap: int, Hq: int, Hkv: int, d: int, seed: int,
                  n_steps: int, B: int = 1):
    """(k_cache, v_cache, q_steps) bf16 CPU tensors:
    k_cache, v_cache [B, Lcap, Hkv, d]; q_steps [n_steps, B, Hq, d]."""
    g = torch.Generator().manual_seed(int(seed))
    k_cache = _draw((B, Lcap, Hkv, d), g)
    v_cache = _draw((B, Lcap, Hkv, d), g)
    q_steps = _draw((n_steps, B, Hq, d), g)
    return k_cache, v_cache, q_steps
