"""fp32 master <-> (bf16 model param, int16 remainder) -- CPU oracle (test only).

"Support store_param_remainders feature from Apex in TE Fused Adam #1408",
Description: with fp32 master params and bf16 model params, keep only the
trailing 16 remainder bits of the master beside the bf16 param and rebuild the
fp32 master from the pair, halving master-parameter memory.

The page fixes no rounding rule.  Reading taken (the only one under which the
sign of the int16 alone says whether the bf16 half was rounded up, giving a
bijection on every bit pattern but the NaNs, see below):

  split:  lo  = bits & 0xFFFF
          hi  = ((bits >> 16) + (lo >= 0x8000)) mod 2**16
          rem = lo reinterpreted as int16
  join:   bits = ((hi - (rem < 0)) mod 2**16) << 16 | (rem as uint16)

``hi`` is therefore the bf16 nearest to the master, ties rounded away from
zero (the increment acts on the magnitude bits).  Everything is integer bit
manipulation: no float arithmetic is involved, so zeros, -0, subnormals and
inf round-trip bit for bit.  (The same page reports NaNs when a parameter
starts at exactly zero in one implementation; this formulation has no such
case.)

A NaN master is first replaced by the quiet NaN 0x7FC00000, so it is stored as
bf16 0x7FC0 (a NaN) with remainder 0 and rebuilt as that NaN.  The bf16 half is
the model's parameter, the master rounded to bf16, and the bf16 nearest to a
NaN is a NaN; left to the increment, the NaN masters 0x7FFF8000-0x7FFFFFFF and
0xFFFF8000-0xFFFFFFFF would carry out of the 16-bit half and read as -0.0 /
+0.0 -- among them 0x7FFFFFFF, the NaN a GPU's arithmetic returns.  join(split(x))
is x for every master but a NaN, and a NaN for a NaN.
"""

from __future__ import annotations

import numpy as np

QNAN = np.uint32(0x7FC00000)   # the quiet NaN a NaN master is stored as


def split(master: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 master (float32 array, or its uint32 bits) -> (bf16 bits uint16, int16 remainder)."""
    bits = np.asarray(master)
    bits = bits.view(np.uint32) if bits.dtype == np.float32 else bits.astype(np.uint32)
    bits = np.where((bits & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000), QNAN, bits)
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
