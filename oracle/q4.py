"""AdamW with 4-bit blockwise-quantised moments -- CPU oracle (test only).

The 8-bit method of ``oracle.q8`` (bitsandbytes PR #2040's blockwise 2-state
step: update with the dequantised moments, then re-quantise m' and v' per
block) with 4-bit codes and smaller blocks.  The pages name torchao's
AdamW4bit ("4 bit Adam should support non constant lr") without its format;
the reading taken (see ``qmap``): blocks of 128 elements with one fp32 absmax
per block and per moment, m on the 16-entry signed dynamic map, v on the
16-entry linear map without zero.

Storage: two codes per byte, the even element in the low nibble and the odd
one in the high nibble; a tensor of n elements holds ceil(n/2) bytes per
moment (an odd n leaves the last high nibble 0).

Step, per block, in the order written: dequantise (``map[code] * absmax``),
update exactly as ``adamw.elementwise_f32``, absmax of m' and v' over float32
bit patterns, normalise ``x = m' * fl(1/A)`` (2**64 scaling below 2**-64) and
take the nearest code (exact ties to the lower code, NaN to code 0).  An
all-zero block stores absmax 0 and the map's zero code, or code 0 for the v
map, which has no zero.
"""

from __future__ import annotations

import numpy as np

from . import adamw, q8
from . import qmap as qm

F32 = np.float32
BLOCK = 128


def pack(codes: np.ndarray) -> np.ndarray:
    """uint8 codes (each < 16) -> ceil(n/2) bytes, even element in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    if np.any(c > 15):
        raise ValueError("4-bit codes must be < 16")
    if c.size % 2:
        c = np.concatenate([c, np.zeros(1, np.uint8)])
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8)


def unpack(packed: np.ndarray, n: int) -> np.ndarray:
    """The first n codes of a packed array."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.size * 2, dtype=np.uint8)
    out[0::2] = b & 0x0F
    out[1::2] = b >> 4
    return out[:n]


class Maps4:
    """The two 4-bit code maps and their thresholds."""

    def __init__(self):
        self.smap = qm.signed_map4()
        self.umap = qm.unsigned_map4()
        self.sthr = qm.thresholds(self.smap)
        self.uthr = qm.thresholds(self.umap)


def quantize_blockwise(x: np.ndarray, table: np.ndarray, thr: np.ndarray,
                       block: int = BLOCK, rule: str = "reciprocal") -> tuple[np.ndarray, np.ndarray]:
    """float32 state -> (codes, one per element, < 16; float32 absmax per block)."""
    x = np.asarray(x, dtype=F32)
    nb = q8.n_blocks(x.size, block)
    codes = np.empty(x.size, dtype=np.uint8)
    amax = np.empty(nb, dtype=F32)
    z = qm.empty_block_code(table)
    for b in range(nb):
        xb = x[b * block:(b + 1) * block]
        a = q8.absmax_bits(xb)
        amax[b] = a
        if a == 0:
            codes[b * block:(b + 1) * block] = z
        else:
            codes[b * block:(b + 1) * block] = qm.quantize(q8.normalise(xb, a, rule), table, thr)
    return codes, amax


def dequantize(packed: np.ndarray, absmax: np.ndarray, table: np.ndarray, n: int,
               block: int = BLOCK) -> np.ndarray:
    return q8.dequantize(unpack(packed, n), absmax, table, block)


def step_f32(p, g, pm, pv, am, av, *, lr, beta1, beta2, eps, wd, t, grad_scale=None,
             maps: Maps4 | None = None, rule: str = "reciprocal") -> bool:
    """One strict-fp32 4-bit-state AdamW step on one flat tensor, in place.

    ``pm``, ``pv`` packed uint8 [ceil(n/2)]; ``am``, ``av`` float32 [ceil(n/128)].
    """
    if grad_scale is not None and adamw.any_nonfinite([g]):
        return False
    maps = maps or Maps4()
    n = np.asarray(p).size
    s = adamw.f32_scalars(lr=lr, beta1=beta1, beta2=beta2, eps=eps, t=t, grad_scale=grad_scale)
    m = dequantize(pm, am, maps.smap, n)
    v = dequantize(pv, av, maps.umap, n)
    p1, m1, v1 = adamw.elementwise_f32(p, g, m, v, s, adamw.decay_f32(s.lr, wd))
    cm1, am1 = quantize_blockwise(m1, maps.smap, maps.sthr, rule=rule)
    cv1, av1 = quantize_blockwise(v1, maps.umap, maps.uthr, rule=rule)
    p[...] = p1
    pm[...] = pack(cm1)
    pv[...] = pack(cv1)
    am[...] = am1
    av[...] = av1
    return True


def step_fp64(p, g, m_state, v_state, *, lr, beta1, beta2, eps, wd, t, grad_scale=None,
              maps: Maps4 | None = None):
    """The same method in float64 (closed-form checks); states are
    ``(packed codes, absmax)`` pairs.  Returns ``(p', (pm', am'), (pv', av'))``."""
    maps = maps or Maps4()
    n = np.asarray(p).size
    cm, am = m_state
    cv, av = v_state
    idx = np.arange(n) // BLOCK
    m = maps.smap.astype(np.float64)[unpack(cm, n)] * np.asarray(am, np.float64)[idx]
    v = maps.umap.astype(np.float64)[unpack(cv, n)] * np.asarray(av, np.float64)[idx]
    x = adamw.Tensor(p=np.asarray(p, np.float64).copy(), g=np.asarray(g, np.float64),
                     m=m, v=v, wd=wd)
    adamw.step_fp64([x], lr=lr, beta1=beta1, beta2=beta2, eps=eps, t=t, grad_scale=grad_scale)
    out = []
    for st, table in ((x.m, maps.smap), (x.v, maps.umap)):
        nb = q8.n_blocks(n, BLOCK)
        codes = np.empty(n, np.uint8)
        amax = np.empty(nb, F32)
        for b in range(nb):
            sb = st[b * BLOCK:(b + 1) * BLOCK]
            a = np.abs(sb).max()
            amax[b] = F32(a)
            codes[b * BLOCK:(b + 1) * BLOCK] = (
                qm.empty_block_code(table) if a == 0 else qm.quantize((sb / a).astype(F32), table))
        out.append((pack(codes), amax))
    return x.p, out[0], out[1]
