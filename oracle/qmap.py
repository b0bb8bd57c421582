"""8-bit and 4-bit code maps and nearest-code quantisation -- CPU oracle.

Test infrastructure only.  **parity unpinned**: the pages never print the code
map.  The bitsandbytes PR ("Fix decoupled weight decay ordering ...") only
names the 8-bit blockwise 2-state kernel and its per-step state quantisation
error (6.6e-4); the workload fixes "a signed 256-entry dynamic exponent code
map in [-1,1]" for m and an unsigned one for v, with one fp32 absmax per
256-element block.  The map is built here from the published description of
dynamic (tree) quantisation -- Dettmers et al., "8-bit Optimizers via
Block-wise Quantization" (arXiv:2110.02861), sec. 2 -- read as: after the sign
bit, a run of E zero bits gives a decimal exponent 10**-E, a 1 bit ends the
run, and the F bits after it split the interval [0.1, 1] into 2**F equal
bins whose centres are the representable fractions.

Concrete construction (this repository's reading, written from that text):

  signed map   (m):  7 magnitude bits; E = 0..6 zero bits, F = 6 - E fraction
                     bits, 2**F values per exponent and per sign:
                     +-10**-E * (0.1 + (k + 1/2) * 0.9 / 2**F)
                     -> 127 magnitudes x 2 signs = 254 values, plus 0 and +1.0.
  unsigned map (v):  the sign bit becomes one more fraction bit:
                     F = 7 - E, E = 0..6 -> 254 positive values, plus 0, +1.0.

Each value is the exact rational rounded once to the nearest float32; the 256
values are sorted ascending and the code of a value is its index.  Exact 0
makes an all-zero state quantise exactly (the first-step closed form of the
bitsandbytes PR relies on that) and exact 1.0 keeps the block maximum exact.

4-bit maps (**parity unpinned** too): the pages name torchao's AdamW4bit
("4 bit Adam should support non constant lr"; the torchtitan job config of
"Adam-mini <> DTensor") but print no format.  Reading taken: the format of
Li, Chen, Zhu, "Memory Efficient Optimizers with 4-bit States" (NeurIPS
2023), which that optimizer implements -- the first moment on the same
dynamic tree at 4 bits (3 magnitude bits: E = 0..2, F = 2 - E, both signs,
plus 0 and +1.0: 16 values), the second moment on the linear map without
zero, k/16 for k = 1..16 (zero is left out because a v quantised to 0 turns
the update into m/eps -- the paper's zero-point problem).

Quantisation rule (also a reading: the pages are silent): the code of a
float32 ``x`` is the index of the nearest map value, an exact tie going to the
lower index; NaN quantises to code 0.  ``quantize_bruteforce`` is that rule
written out; ``quantize`` is the same rule through per-gap thresholds
(``thresholds``), ``code = #{k : thr[k] <= x}``, used for large arrays.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

F32 = np.float32


def _round_to_f32(q: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) float32 of an exact rational."""
    c = F32(float(q))  # float64 rounding, then float32: may double-round ...
    best = None
    for cand in (np.nextafter(c, F32(-np.inf)), c, np.nextafter(c, F32(np.inf))):
        d = abs(Fraction(float(cand)) - q)  # ... so pick the nearest neighbour exactly
        key = (d, int(np.asarray(cand).view(np.uint32)) & 1)  # tie -> even mantissa
        if best is None or key < best[0]:
            best = (key, cand)
    return F32(best[1])


def _dynamic_values(frac_bits_at_e0: int, signed: bool, n_exp: int = 7,
                    size: int = 256) -> np.ndarray:
    vals = [Fraction(0), Fraction(1)]
    for e in range(n_exp):
        f = frac_bits_at_e0 - e
        n = 2 ** f
        for k in range(n):
            mag = (Fraction(1, 10) + Fraction(2 * k + 1, 2 * n) * Fraction(9, 10)) / 10 ** e
            vals.append(mag)
            if signed:
                vals.append(-mag)
    out = np.array(sorted(_round_to_f32(q) for q in vals), dtype=F32)
    if out.size != size or np.unique(out).size != size:
        raise AssertionError(f"code map must hold {size} distinct values")
    return out


def signed_map() -> np.ndarray:
    """256 sorted float32 values in [-1, 1] for the first moment."""
    return _dynamic_values(6, signed=True)


def unsigned_map() -> np.ndarray:
    """256 sorted float32 values in [0, 1] for the second moment."""
    return _dynamic_values(7, signed=False)


def signed_map4() -> np.ndarray:
    """16 sorted float32 values in [-1, 1] for the 4-bit first moment."""
    return _dynamic_values(2, signed=True, n_exp=3, size=16)


def unsigned_map4() -> np.ndarray:
    """k/16 for k = 1..16 (no zero), the 4-bit second-moment map."""
    return (np.arange(1, 17, dtype=np.float64) / 16).astype(F32)


def zero_code(qmap: np.ndarray) -> int:
    """Index of the exact 0.0 entry."""
    (idx,) = np.nonzero(qmap == 0)
    return int(idx[0])


def empty_block_code(qmap: np.ndarray) -> int:
    """Code stored for an all-zero block (absmax 0): the zero entry, or code 0
    for a map without one (it dequantises to 0 through the zero absmax)."""
    (idx,) = np.nonzero(qmap == 0)
    return int(idx[0]) if idx.size else 0


def quantize_bruteforce(x: np.ndarray, qmap: np.ndarray) -> np.ndarray:
    """Nearest-code rule written out: argmin_k |x - map[k]| (exact), lowest k on ties."""
    x = np.asarray(x, dtype=F32).ravel()
    codes = np.zeros(x.size, dtype=np.uint8)
    table = [Fraction(float(q)) for q in qmap]
    for i, xi in enumerate(x):
        if np.isnan(xi):
            codes[i] = 0
            continue
        xf = Fraction(float(xi))
        best_k, best_d = 0, None
        for k, q in enumerate(table):
            d = abs(xf - q)
            if best_d is None or d < best_d:
                best_k, best_d = k, d
        codes[i] = best_k
    return codes


def thresholds(qmap: np.ndarray) -> np.ndarray:
    """thr[k] = the smallest float32 strictly above the exact midpoint of map[k], map[k+1].

    A float32 ``x`` is strictly nearer to ``map[k+1]`` than to ``map[k]``
    exactly when ``x > (map[k] + map[k+1]) / 2``, i.e. when ``x >= thr[k]``.
    The midpoint is exact in float64: both neighbours are float32 of
    magnitude <= 1 whose exponents differ by fewer than 29 binades.
    """
    q = qmap.astype(np.float64)
    out = np.empty(q.size - 1, dtype=F32)
    for k in range(q.size - 1):
        mid = (q[k] + q[k + 1]) / 2.0
        assert Fraction(mid) == (Fraction(q[k]) + Fraction(q[k + 1])) / 2
        c = F32(mid)
        if float(c) <= mid:
            c = np.nextafter(c, F32(np.inf))
        out[k] = c
    return out


def quantize(x: np.ndarray, qmap: np.ndarray, thr: np.ndarray | None = None) -> np.ndarray:
    """Nearest-code rule via thresholds: code = #{k : thr[k] <= x}; NaN -> 0."""
    if thr is None:
        thr = thresholds(qmap)
    x = np.asarray(x, dtype=F32)
    codes = np.searchsorted(thr, x, side="right").astype(np.uint8)
    codes[np.isnan(x)] = 0
    return codes
