"""Plain, slow, fp64 CPU oracle for causal bifocal-RoPE attention (Jet-Long).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA path (no
kernels, headers, tables or constant generators); the only thing both sides
share is the seeded input generator, which holds none of the method's
arithmetic.

Parity status of each function is stated in ``oracle/bifocal.py``'s header.
"""

from .bifocal import (  # noqa: F401
    group_size,
    alias,
    rope_frequencies,
    rope_cos_sin,
    rope_rotate,
    round_to_bf16,
    bifocal_prefill,
    bifocal_prefill_three_pass,
    bifocal_decode,
    bifocal_prefill_chunk,
)
