"""AdamW with 8-bit blockwise-quantised moments -- CPU oracle (test only).

"Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
(bitsandbytes PR #2040), PR description: the 8-bit blockwise 2-state step
applies the same decoupled AdamW update as the 32-bit one; its moments are
stored quantised, an all-zero state quantises exactly, and the per-step state
quantisation error (6.6e-4) is the method's own cost.  Block size (256
elements, one fp32 absmax per block and per moment), the signed map for m and
the unsigned map for v come from the workload definition; the maps themselves
are in ``qmap`` (parity unpinned there).

Step, per block of 256 consecutive elements of one tensor (the last block of a
tensor may be partial), in the order written:

  dequantise   m = smap[cm] * Am          v = umap[cv] * Av
  update       m', v', p'  exactly as ``adamw.elementwise_f32`` (fp32 mode)
               -- the parameter update uses m', v' *before* re-quantisation
  absmax       Am' = max |m'|,  Av' = max |v'|   (max of the float32 bit
               patterns with the sign cleared: exact and order-free; equals
               the float maximum for non-NaN data)
  requantise   x = m' * fl(1/Am')   (Am' == 0: the zero code), cm' = nearest code of x
               y = v' * fl(1/Av')   likewise with the unsigned map
               -- the ratio is formed with the block's reciprocal rounded once
               and one multiply per element; when the absmax is below 2**-64
               both factors are first scaled by 2**64 (exact), so that the
               reciprocal cannot overflow

Readings (the pages are silent): an all-zero block stores absmax 0 and the
zero code; nearest-code ties go to the lower code; v uses its own absmax
``max v'`` with the unsigned map; the normalised value is ``m' * fl(1/absmax)``
(one reciprocal per block), not a per-element division.
"""

from __future__ import annotations

import numpy as np

from . import adamw, qmap as qm

F32 = np.float32
BLOCK = 256


def n_blocks(numel: int, block: int = BLOCK) -> int:
    return (numel + block - 1) // block


def absmax_bits(x: np.ndarray) -> np.float32:
    """max |x| taken over float32 bit patterns with the sign bit cleared."""
    b = np.asarray(x, dtype=F32).view(np.uint32) & np.uint32(0x7FFFFFFF)
    return b.max().view(F32) if b.size else F32(0)


def dequantize(codes: np.ndarray, absmax: np.ndarray, table: np.ndarray,
               block: int = BLOCK) -> np.ndarray:
    """float32 state from codes: table[code] * absmax[block of the element]."""
    codes = np.asarray(codes)
    idx = np.arange(codes.size) // block
    return (table[codes] * np.asarray(absmax, dtype=F32)[idx]).astype(F32)


SMALL = F32(2.0 ** -64)
SCALE = F32(2.0 ** 64)


def normalise(xb: np.ndarray, a: np.float32, rule: str = "reciprocal") -> np.ndarray:
    """x * fl(1/a), with x and a first scaled by 2**64 when a < 2**-64 (exact scalings).

    ``rule="division"`` is the plain ratio fl(x / a), one correctly rounded
    division per element (never out of range: |x| <= a).  The library uses
    the reciprocal form, a reading taken for speed; the tests bound how far it
    can move a code from the division form.
    """
    if rule == "division":
        return (np.asarray(xb, dtype=F32) / F32(a)).astype(F32)
    s = SCALE if a < SMALL else F32(1.0)
    y = F32(1.0) / F32(a * s)
    return (np.asarray(xb, dtype=F32) * s) * y


def quantize_blockwise(x: np.ndarray, table: np.ndarray, thr: np.ndarray,
                       block: int = BLOCK, rule: str = "reciprocal") -> tuple[np.ndarray, np.ndarray]:
    """float32 state -> (uint8 codes, float32 absmax per block)."""
    x = np.asarray(x, dtype=F32)
    nb = n_blocks(x.size, block)
    codes = np.empty(x.size, dtype=np.uint8)
    amax = np.empty(nb, dtype=F32)
    z = qm.zero_code(table)
    for b in range(nb):
        xb = x[b * block:(b + 1) * block]
        a = absmax_bits(xb)
        amax[b] = a
        if a == 0:
            codes[b * block:(b + 1) * block] = z
        else:
            codes[b * block:(b + 1) * block] = qm.quantize(normalise(xb, a, rule), table, thr)
    return codes, amax


class Maps:
    """The two code maps and their thresholds."""

    def __init__(self, smap: np.ndarray | None = None, umap: np.ndarray | None = None):
        self.smap = qm.signed_map() if smap is None else np.asarray(smap, dtype=F32)
        self.umap = qm.unsigned_map() if umap is None else np.asarray(umap, dtype=F32)
        self.sthr = qm.thresholds(self.smap)
        self.uthr = qm.thresholds(self.umap)


def step_f32(p, g, cm, cv, am, av, *, lr, beta1, beta2, eps, wd, t,
             grad_scale=None, maps: Maps | None = None, block: int = BLOCK,
             rule: str = "reciprocal") -> bool:
    """One strict-fp32 8-bit-state AdamW step on one flat tensor, in place.

    ``p`` float32 [n]; ``g`` raw grads [n]; ``cm``, ``cv`` uint8 codes [n];
    ``am``, ``av`` float32 absmax [ceil(n/block)].  Returns False (nothing
    changed) when a grad scale is given and a raw grad is non-finite.
    ``rule`` selects the normalisation (``normalise``).
    """
    if grad_scale is not None and adamw.any_nonfinite([g]):
        return False
    maps = maps or Maps()
    s = adamw.f32_scalars(lr=lr, beta1=beta1, beta2=beta2, eps=eps, t=t,
                          grad_scale=grad_scale)
    m = dequantize(cm, am, maps.smap, block)
    v = dequantize(cv, av, maps.umap, block)
    p1, m1, v1 = adamw.elementwise_f32(p, g, m, v, s, adamw.decay_f32(s.lr, wd))
    cm1, am1 = quantize_blockwise(m1, maps.smap, maps.sthr, block, rule)
    cv1, av1 = quantize_blockwise(v1, maps.umap, maps.uthr, block, rule)
    p[...] = p1
    cm[...] = cm1
    cv[...] = cv1
    am[...] = am1
    av[...] = av1
    return True


def step_fp64(p, g, m_state, v_state, *, lr, beta1, beta2, eps, wd, t,
              grad_scale=None, maps: Maps | None = None, block: int = BLOCK):
    """The same method in float64, for closed-form checks.

    ``m_state`` / ``v_state`` are ``(codes, absmax)`` pairs; dequantisation,
    update and the ratio ``x = m'/A`` are float64, the nearest code is chosen
    for ``x`` rounded to float32.  Returns ``(p', (cm', am'), (cv', av'))`` with
    p' in float64 and absmax rounded to float32 for storage.
    """
    maps = maps or Maps()
    cm, am = m_state
    cv, av = v_state
    idx = np.arange(np.asarray(p).size) // block
    m = maps.smap.astype(np.float64)[cm] * np.asarray(am, np.float64)[idx]
    v = maps.umap.astype(np.float64)[cv] * np.asarray(av, np.float64)[idx]
    x = adamw.Tensor(p=np.asarray(p, np.float64).copy(), g=np.asarray(g, np.float64),
                     m=m, v=v, wd=wd)
    adamw.step_fp64([x], lr=lr, beta1=beta1, beta2=beta2, eps=eps, t=t,
                    grad_scale=grad_scale)
    out = []
    for st, table in ((x.m, maps.smap), (x.v, maps.umap)):
        nb = n_blocks(st.size, block)
        codes = np.empty(st.size, np.uint8)
        amax = np.empty(nb, F32)
        for b in range(nb):
            sb = st[b * block:(b + 1) * block]
            a = np.abs(sb).max()
            amax[b] = F32(a)
            codes[b * block:(b + 1) * block] = (
                qm.zero_code(table) if a == 0 else qm.quantize((sb / a).astype(F32), table))
        out.append((codes, amax))
    return x.p, out[0], out[1]
