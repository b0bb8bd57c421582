"""CPU oracle for the fused AdamW step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct numpy implementations of what the GPU path
computes. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py`` may import anything from here. The GPU library
never imports, links or calls this package, and this package imports nothing
from the GPU library: the two share no code.

Modules
-------
adamw      decoupled-weight-decay AdamW step, fp64 definition and a strict-fp32
           mode with one rounding per written operation (AMP unscale and the
           found_inf skip included).
ademamix   AdEMAMix (fast and slow EMA) with the same decoupled decay, both modes.
lion       Lion (sign update, one state) with decay before the update, both modes.
coupled    momentum, RMSprop and Adagrad (one state) with coupled L2 decay, both modes.
mini       Adam-mini: one second moment per block (element, head or tensor), both modes.
remainder  fp32 master <-> (bf16 model param, int16 remainder) split and join.
qmap       the dynamic-exponent 8-bit code maps, their decision thresholds and
           nearest-code quantisation.
q8         the AdamW step with 8-bit blockwise-quantised moments.
q4         the same step with 4-bit codes (two per byte) and 128-element blocks.

Pins (what ties each function to something other than itself) live in
``tests/test_oracle_*.py``.  One function is **parity unpinned** by the pages:
the contents of the 8-bit and 4-bit code maps (``qmap.signed_map`` /
``qmap.unsigned_map``, ``qmap.signed_map4`` / ``qmap.unsigned_map4``); the pages never
print a map, so only its structural
invariants and the quantiser built on top of it are pinned.
"""

from . import adamw, ademamix, coupled, lion, mini, remainder, qmap, q4, q8  # noqa: F401
