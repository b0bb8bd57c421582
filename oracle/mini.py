"""Adam-mini -- CPU oracle (test infrastructure only).

"Adam-mini <> DTensor", the ``AdamWMini`` listing: every tensor keeps a full
first moment ``m``, but its second moment is shared by blocks of contiguous
elements -- one value per element for embeddings and the output layer (the
AdamW branch), one per attention head for the query and key weights (blocks
of ``dim*dim/n_heads`` elements), one per tensor for everything else.  Here a
tensor carries its block length ``block`` (1, a head size, or numel) and
``v`` holds ``numel/block`` values; which block length a tensor gets is the
caller's choice of partition, as the listing makes it from parameter names.

Per tensor, in the listing's order (t = the 1-based step):

  g      = g_raw [/ grad_scale]
  v_b    = b2*v_b + (1-b2) * mean over block b of g*g
  p      = p * (1 - lr*wd)                   only when wd > 0
  m      = b1*m + (1-b1)*g                   (the listing writes lerp)
  h_b    = sqrt(v_b) / sqrt(1 - b2^t) + eps
  p      = p - lr * m * ((1/(1 - b1^t)) / h_b)

For block 1 this is the AdamW branch (``p += -(lr/bc1) * m / h``), the same
value in exact arithmetic.  The AMP skip is ``oracle.adamw``'s.

``step_f32``: the strict-fp32 specification, one rounding per operation,
with the bias corrections of ``adamw.f32_scalars`` (rbc1 = fl(1/bc1)).  A
tensor with block 1 follows the AdamW branch as the listing writes it
(``addcdiv``): exactly ``adamw.elementwise_f32``.  Blocks longer than 1:

  g = g_raw [* inv_scale]
  S_b = sum of g*g over the block in float64 (each square is exact in float64;
        the sum may be taken in any order), mean_b = fl32(S_b / block)
  v_b' = b2*v_b + omb2*mean_b
  h_b = sqrt(v_b')*inv_sqrt_bc2 + eps ;  r_b = rbc1 / h_b
  m' = b1*m + omb1*g ;  u = m'*r_b ;  p' = p*decay - lr*u
       (decay = fl(1 - fl(lr*wd)) when wd > 0, else the parameter is not scaled)

The float64 sum is the one place where rounding order is left open: two
correct implementations agree on ``mean_b`` except when the exact mean lies
within about 1e-16 (relative) of a float32 rounding boundary.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import adamw as A

F32 = np.float32
F64 = np.float64


@dataclass
class Tensor:
    p: np.ndarray
    g: np.ndarray
    m: np.ndarray
    v: np.ndarray          # numel // block values
    wd: float
    block: int


def _blocks(x: np.ndarray, block: int) -> np.ndarray:
    n = x.size
    if block < 1 or n % block:
        raise ValueError("block must divide numel")
    return x.reshape(n // block, block)


def step_fp64(tensors: list[Tensor], *, lr, beta1, beta2, eps, t: int,
              grad_scale=None) -> bool:
    """One Adam-mini step in float64, in place."""
    if grad_scale is not None and A.any_nonfinite([x.g for x in tensors]):
        return False
    b1, b2, lr, eps = F64(beta1), F64(beta2), F64(lr), F64(eps)
    bc1 = 1 - b1 ** t
    bc2 = 1 - b2 ** t
    for x in tensors:
        if x.p.size == 0:
            continue
        g = np.asarray(x.g, dtype=F64)
        if grad_scale is not None:
            g = g / F64(grad_scale)
        gb = _blocks(g, x.block)
        x.v[...] = b2 * x.v + (1 - b2) * np.mean(gb * gb, axis=1)
        if x.wd > 0:
            x.p[...] = x.p * (1 - lr * F64(x.wd))
        x.m[...] = b1 * x.m + (1 - b1) * g
        h = np.sqrt(x.v) / np.sqrt(bc2) + eps
        step = (1 / bc1) / h
        x.p[...] = x.p - lr * (_blocks(x.m, x.block) * step[:, None]).ravel()
    return True


def block_mean_sq(g32: np.ndarray, block: int) -> np.ndarray:
    """fl32(S_b / block), S_b the float64 sum of the exact squares of a block."""
    gb = _blocks(np.asarray(g32, dtype=F32).astype(F64), block)
    return (np.sum(gb * gb, axis=1) / F64(block)).astype(F32)


def block_sum_sq(g32: np.ndarray) -> np.float64:
    """The float64 sum of the exact squares of some float32 values.  The order
    of a block's sum is free, so a block too large to hold at once is summed
    piece by piece: S_b = the float64 sum of its pieces' block_sum_sq."""
    x = np.asarray(g32, dtype=F32).astype(F64)
    return F64(np.sum(x * x))


def mean_from_sum(s_b: np.float64, length: int) -> np.float32:
    """mean_b = fl32(S_b / block length)."""
    return F32(F64(s_b) / F64(length))


def step_f32(tensors: list[Tensor], *, lr, beta1, beta2, eps, t: int,
             grad_scale=None, means: list | None = None) -> bool:
    """One strict-fp32 Adam-mini step, in place (float32 p, m, v).

    ``means`` (optional, per tensor: None or float32 block means from
    ``mean_from_sum``) stands in for the block means of ``x.g``: it lets a
    caller follow a sample of one huge block, whose mean it summed piece by
    piece, with ``x.p``, ``x.g``, ``x.m`` holding only the sampled elements
    (``x.block`` = the sample's length).  Without a grad scale only."""
    if grad_scale is not None and A.any_nonfinite([x.g for x in tensors]):
        return False
    s = A.f32_scalars(lr=lr, beta1=beta1, beta2=beta2, eps=eps, t=t, grad_scale=grad_scale)
    bc1, _ = A.bias_corrections(float(F32(beta1)), float(F32(beta2)), t)
    rbc1 = F32(F32(1.0) / F32(bc1))
    for i, x in enumerate(tensors):
        if x.p.size == 0:
            continue
        decay = A.decay_f32(s.lr, x.wd) if x.wd > 0 else F32(1.0)
        given = None if means is None else means[i]
        if x.block == 1 and given is None:
            p1, m1, v1 = A.elementwise_f32(x.p, x.g, x.m, x.v, s, decay)
            x.p[...], x.m[...], x.v[...] = p1, m1, v1
            continue
        g = np.asarray(x.g).astype(F32)
        if s.inv_scale is not None:
            g = g * s.inv_scale
        if given is not None and s.inv_scale is not None:
            raise ValueError("precomputed block means are for unscaled grads")
        mean = block_mean_sq(g, x.block) if given is None else np.asarray(given, dtype=F32)
        v1 = s.b2 * x.v + s.omb2 * mean
        h = np.sqrt(v1) * s.inv_sqrt_bc2 + s.eps
        r = rbc1 / h
        m1 = s.b1 * x.m + s.omb1 * g
        u = (_blocks(m1, x.block) * r[:, None]).ravel()
        x.p[...] = (x.p * decay - s.lr * u).astype(F32)
        x.m[...] = m1.astype(F32)
        x.v[...] = v1.astype(F32)
    return True
