"""Lion with decoupled weight decay -- CPU oracle (test infrastructure only).

"Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
(bitsandbytes PR #2040), reviewer's note on the 1-state kernels: Lion applies
decoupled decay to the parameter *before* its sign update -- the ordering the
PR establishes for AdamW.  The update itself is restated from Chen et al.,
"Symbolic Discovery of Optimization Algorithms" (arXiv:2302.06675):

  c  = b1*m + (1-b1)*g             interpolation that decides the direction
  p  = p*(1 - lr*wd) - lr*sign(c)
  m  = b2*m + (1-b2)*g             the state keeps the b2 EMA

sign(0) = 0; a NaN c counts as 0 (reading: the page gives no rule; with the
AMP skip a NaN never reaches the update).  No bias correction.  Grad unscale
and the non-finite skip are those of ``oracle.adamw``.

``step_f32`` is the strict-fp32 specification, one rounding per operation in
this order: g [* inv_scale]; c = b1*m + omb1*g; s = sign(c);
p' = p*decay - lr*s; m' = b2*m + omb2*g.
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
    wd: float


def sign(c: np.ndarray) -> np.ndarray:
    """+1, -1 or 0 (zero and NaN give 0), in c's dtype."""
    c = np.asarray(c)
    return ((c > 0).astype(c.dtype) - (c < 0).astype(c.dtype)).astype(c.dtype)


def step_fp64(tensors: list[Tensor], *, lr, beta1, beta2, grad_scale=None,
              decay_after=False) -> bool:
    """One Lion step in float64, in place.  ``decay_after`` is the wrong ordering
    (kept only so the tests can show they reject it)."""
    if grad_scale is not None and A.any_nonfinite([x.g for x in tensors]):
        return False
    b1, b2, lr = F64(beta1), F64(beta2), F64(lr)
    for x in tensors:
        g = np.asarray(x.g, dtype=F64)
        if grad_scale is not None:
            g = g / F64(grad_scale)
        c = b1 * x.m + (1 - b1) * g
        decay = 1 - lr * F64(x.wd)
        if decay_after:
            x.p[...] = (x.p - lr * sign(c)) * decay
        else:
            x.p[...] = x.p * decay - lr * sign(c)
        x.m[...] = b2 * x.m + (1 - b2) * g
    return True


def step_f32(tensors: list[Tensor], *, lr, beta1, beta2, grad_scale=None) -> bool:
    """One strict-fp32 Lion step, in place (float32 p, m)."""
    if grad_scale is not None and A.any_nonfinite([x.g for x in tensors]):
        return False
    b1, b2, lr32 = F32(beta1), F32(beta2), F32(lr)
    omb1, omb2 = F32(F32(1.0) - b1), F32(F32(1.0) - b2)
    inv = None if grad_scale is None else F32(F32(1.0) / F32(grad_scale))
    for x in tensors:
        decay = A.decay_f32(lr32, x.wd)
        g = np.asarray(x.g).astype(F32)
        if inv is not None:
            g = g * inv
        c = b1 * x.m + omb1 * g
        x.p[...] = (x.p * decay - lr32 * sign(c)).astype(F32)
        x.m[...] = (b2 * x.m + omb2 * g).astype(F32)
    return True
