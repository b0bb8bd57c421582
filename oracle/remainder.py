"""fp32 master <-> (bf16 model param, int16 remainder) -- CPU oracle (test only).

"Support store_param_remainders feature from Apex in TE Fused Adam #1408",
Description: with fp32 master params and bf16 model params, keep only the
trailing 16 remainder bits of the master beside the bf16 param and rebuild the
fp32 master from the pair, halving master-parameter memory.

The page fixes no rounding rule.  Reading taken (the only one under which the
sign of the int16 alone says whether the bf16 half was rounded up, giving a
bijection on all 2**32 bit patterns):

  split:  lo  = bits & 0xFFFF
          hi  = ((bits >> 16) + (lo >= 0x8000)) mod 2**16
          rem = lo reinterpreted as int16
  join:   bits = ((hi - (rem < 0)) mod 2**16) << 16 | (rem as uint16)

``hi`` is therefore the bf16 nearest to the master, ties rounded away from
zero (the increment acts on the magnitude bits).  Everything is integer bit
manipulation: no float arithmetic is involved, so zeros, -0, subnormals, inf
and NaN all round-trip.  (The same page reports NaNs when a parameter starts at
exactly zero in one implementation; this formulation has no such case.)
For the NaN masters 0x7FFF8000-0x7FFFFFFF and 0xFFFF8000-0xFFFFFFFF the
increment carries out of the 16-bit half, so ``hi`` reads as -0.0 / +0.0; the
master is still rebuilt exactly by ``join``.
"""

from __future__ import annotations

import numpy as np


def split(master: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 master (float32 array, or its uint32 bits) -> (bf16 bits uint16, int16 remainder)."""
    bits = np.asarray(master)
    bits = bits.view(np.uint32) if bits.dtype == np.float32 else bits.astype(np.uint32)
    lo = bits & np.uint32(0xFFFF)
    hi = ((bits >> np.uint32(16)) + (lo >= np.uint32(0x8000)).astype(np.uint32)) & np.uint32(0xFFFF)
    return hi.astype(np.uint16), lo.astype(np.uint16).view(np.int16)


def join(hi: np.ndarray, rem: np.ndarray) -> np.ndarray:
    """(bf16 bits uint16, int16 remainder) -> fp32 master as float32."""
    hi = np.asarray(hi).astype(np.uint32)
    rem = np.asarray(rem, dtype=np.int16)
    top = (hi - (rem < 0).astype(np.uint32)) & np.uint32(0xFFFF)
    bits = (top << np.uint32(16)) | rem.view(np.uint16).astype(np.uint32)
    return bits.astype(np.uint32).view(np.float32)


def bf16_bits_to_f32(hi: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 (exact)."""
    return (np.asarray(hi).astype(np.uint32) << np.uint32(16)).view(np.float32)
