"""AdEMAMix with decoupled weight decay -- CPU oracle (test infrastructure only).

"Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
(bitsandbytes PR #2040), PR description: the AdEMAMix update rule of
Pagliardini et al. (arXiv:2409.03137) takes the decay and the gradient-based
update from the same previous parameter, exactly like AdamW, and one step from
a zero state reduces to the AdamW closed form with ``alpha*(1-b3)*g`` mixed into
the numerator.  The update restated from that paper (its alpha and beta3
warm-up schedules are the caller's business: this step takes their current
values):

  m1 = b1*m1 + (1-b1)*g          fast EMA, bias-corrected
  m2 = b3*m2 + (1-b3)*g          slow EMA, not bias-corrected
  v  = b2*v  + (1-b2)*g*g
  p  = p*(1 - lr*wd) - lr * (m1/bc1 + alpha*m2) / (sqrt(v)/sqrt(bc2) + eps)

with bc1 = 1 - b1**t, bc2 = 1 - b2**t.  Grad unscale and the non-finite skip are
those of ``oracle.adamw``.

``step_f32`` is the strict-fp32 specification (one rounding per operation, in
this order; scalars as in ``oracle.adamw.f32_scalars``, plus
``rbc1 = fl(1 / fl32(bc1))``, ``omb3 = fl(1 - b3)``):

  g   = g_raw [* inv_scale]
  m1' = b1*m1 + omb1*g
  m2' = b3*m2 + omb3*g
  v'  = b2*v + omb2*(g*g)
  h   = sqrt(v') * inv_sqrt_bc2 + eps
  n   = m1'*rbc1 + alpha*m2'
  u   = n / h
  p'  = p*decay - lr*u
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import adamw as A

F32 = np.float32
F64 = np.float64


@dataclass
class Tensor:
    """One tensor's state: param, grad, fast EMA m1, slow EMA m2, v, weight decay."""

    p: np.ndarray
    g: np.ndarray
    m1: np.ndarray
    m2: np.ndarray
    v: np.ndarray
    wd: float


def step_fp64(tensors: list[Tensor], *, lr, beta1, beta2, beta3, alpha, eps, t,
              grad_scale=None) -> bool:
    """One AdEMAMix step in float64, in place; False (unchanged) on a skipped AMP step."""
    if grad_scale is not None and A.any_nonfinite([x.g for x in tensors]):
        return False
    b1, b2, b3 = F64(beta1), F64(beta2), F64(beta3)
    bc1, sqrt_bc2 = A.bias_corrections(beta1, beta2, t)
    for x in tensors:
        g = np.asarray(x.g, dtype=F64)
        if grad_scale is not None:
            g = g / F64(grad_scale)
        m1 = b1 * x.m1 + (1 - b1) * g
        m2 = b3 * x.m2 + (1 - b3) * g
        v = b2 * x.v + (1 - b2) * g * g
        u = (m1 / F64(bc1) + F64(alpha) * m2) / (np.sqrt(v) / F64(sqrt_bc2) + F64(eps))
        x.p[...] = x.p * (1 - F64(lr) * F64(x.wd)) - F64(lr) * u
        x.m1[...], x.m2[...], x.v[...] = m1, m2, v
    return True


def step_f32(tensors: list[Tensor], *, lr, beta1, beta2, beta3, alpha, eps, t,
             grad_scale=None) -> bool:
    """One strict-fp32 AdEMAMix step, in place (float32 p, m1, m2, v)."""
    if grad_scale is not None and A.any_nonfinite([x.g for x in tensors]):
        return False
    s = A.f32_scalars(lr=lr, beta1=beta1, beta2=beta2, eps=eps, t=t, grad_scale=grad_scale)
    bc1, _ = A.bias_corrections(float(F32(beta1)), float(F32(beta2)), t)
    rbc1 = F32(F32(1.0) / F32(bc1))
    b3 = F32(beta3)
    omb3 = F32(F32(1.0) - b3)
    al = F32(alpha)
    for x in tensors:
        decay = A.decay_f32(s.lr, x.wd)
        g = np.asarray(x.g).astype(F32)
        if s.inv_scale is not None:
            g = g * s.inv_scale
        m1 = s.b1 * x.m1 + s.omb1 * g
        m2 = b3 * x.m2 + omb3 * g
        v = s.b2 * x.v + s.omb2 * (g * g)
        h = np.sqrt(v) * s.inv_sqrt_bc2 + s.eps
        n = m1 * rbc1 + al * m2
        u = n / h
        x.p[...] = (x.p * decay - s.lr * u).astype(F32)
        x.m1[...], x.m2[...], x.v[...] = m1, m2, v
    return True
