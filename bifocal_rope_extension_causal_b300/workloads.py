"""The five named workloads (shapes only; no arithmetic of the method).

Shapes follow the Qwen3 attention layers the Jet-Long pages benchmark on
(32K native window extended to 64K and 128K).
"""

from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    index: int          # also the input seed
    L: int
    Hq: int
    Hkv: int
    d: int
    w_pretrained: int
    w0: int
    theta: float
    B: int = 1


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    index: int
    Lcap: int
    lengths: tuple = field(default_factory=tuple)
    Hq: int = 32
    Hkv: int = 8
    d: int = 128
    w_pretrained: int = 32768
    w0: int = 4096
    theta: float = 1e6
    B: int = 1


TINY = PrefillWorkload("tiny prefill L=256 G=4 (2q/1kv, d=64)", 0, 256, 2, 1, 64, 64, 16, 1e4)
NATIVE_32K = PrefillWorkload("native-window prefill L=32768 G=1 (16q/8kv, d=128)", 1,
                             32768, 16, 8, 128, 32768, 4096, 1e6)
EXT_64K = PrefillWorkload("2x extension prefill L=65536 G=2 (32q/8kv, d=128)", 2,
                          65536, 32, 8, 128, 32768, 4096, 1e6)
EXT_128K = PrefillWorkload("4x extension prefill L=131072 G=4 (32q/8kv, d=128)", 3,
                           131072, 32, 8, 128, 32768, 4096, 1e6)
DECODE = DecodeWorkload("decode against an absolute-position cache, L in {32767, 32769, 65537, 131072}",
                        4, 131072, (32767, 32769, 65537, 131072))

PREFILL_WORKLOADS = (TINY, NATIVE_32K, EXT_64K, EXT_128K)


def prefill_causal_pairs(L: int) -> int:
    """Number of (query, key) pairs with key <= query in one head."""
    return L * (L + 1) // 2


def prefill_flops(w: PrefillWorkload) -> float:
    """Algorithmic FLOPs of one prefill: 4*d per causal pair per query head
    (2*d for the score, 2*d for the value update)."""
    return 4.0 * w.d * prefill_causal_pairs(w.L) * w.Hq * w.B


def decode_bytes(L: int, Hkv: int, d: int, Hq: int, B: int = 1) -> int:
    """Algorithmic HBM bytes of one decode step: every cached K and V row of
    the L positions once (bf16), plus the query in and the output out."""
    return B * (2 * L * Hkv * d * 2 + 2 * Hq * d * 2)
