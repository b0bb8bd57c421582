"""1-state optimizers with coupled L2 decay -- CPU oracle (test infrastructure only).

"Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
(bitsandbytes PR #2040), review of the 1-state kernels: for momentum, RMSprop
and Adagrad the decay is folded into the gradient, ``g = g + p*wd`` when
``wd > 0`` -- coupled L2, so there is no ordering question; the parameter is
never decayed directly.  The page names the three rules but does not write
them out; the plainest reading, taken here, is each rule's textbook form with
one state ``s`` (the form torch.optim's SGD / RMSprop / Adagrad use with no
dampening, no centring, no Nesterov and no lr decay):

  momentum  s = b*s + g                       p = p - lr*s
  rmsprop   s = b*s + (1-b)*g*g               p = p - lr * g / (sqrt(s) + eps)
  adagrad   s = s + g*g                       p = p - lr * g / (sqrt(s) + eps)

with ``g`` the unscaled grad plus ``p*wd`` (the decay term joins the grad
after the AMP unscale, as a fused step sees the grad GradScaler would have
unscaled).  ``wd <= 0`` adds nothing, as the page's condition reads.  No bias
correction; the momentum state starts at 0, so its first step is ``s = g``.
The AMP skip is that of ``oracle.adamw``.

``step_f32`` is the strict-fp32 specification, one rounding per operation:
  g = g_raw [* inv_scale];  g = g + p*wd  (only when wd > 0)
  momentum: s' = b*s + g;                   p' = p - lr*s'
  rmsprop:  s' = b*s + fl(1-b)*(g*g);       p' = p - lr*(g / (sqrt(s') + eps))
  adagrad:  s' = s + g*g;                   p' = p - lr*(g / (sqrt(s') + eps))
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import adamw as A

F32 = np.float32
F64 = np.float64

RULES = ("momentum", "rmsprop", "adagrad")


@dataclass
class Tensor:
    p: np.ndarray
    g: np.ndarray
    s: np.ndarray
    wd: float


def step_fp64(tensors: list[Tensor], *, rule: str, lr, beta=0.0, eps=0.0,
              grad_scale=None, decoupled=False) -> bool:
    """One step in float64, in place.  ``decoupled`` (decay the parameter
    instead of the grad) is a wrong reading kept only for the tests."""
    if rule not in RULES:
        raise ValueError(rule)
    if grad_scale is not None and A.any_nonfinite([x.g for x in tensors]):
        return False
    b, lr, eps = F64(beta), F64(lr), F64(eps)
    for x in tensors:
        g = np.asarray(x.g, dtype=F64)
        if grad_scale is not None:
            g = g / F64(grad_scale)
        wd = F64(x.wd)
        p0 = x.p.copy()
        if wd > 0 and not decoupled:
            g = g + p0 * wd
        if rule == "momentum":
            x.s[...] = b * x.s + g
            d = x.s
        elif rule == "rmsprop":
            x.s[...] = b * x.s + (1 - b) * g * g
            d = g / (np.sqrt(x.s) + eps)
        else:
            x.s[...] = x.s + g * g
            d = g / (np.sqrt(x.s) + eps)
        if wd > 0 and decoupled:
            x.p[...] = p0 * (1 - lr * wd) - lr * d
        else:
            x.p[...] = p0 - lr * d
    return True


def step_f32(tensors: list[Tensor], *, rule: str, lr, beta=0.0, eps=0.0,
             grad_scale=None) -> bool:
    """One strict-fp32 step, in place (float32 p and s)."""
    if rule not in RULES:
        raise ValueError(rule)
    if grad_scale is not None and A.any_nonfinite([x.g for x in tensors]):
        return False
    b, lr32, eps32 = F32(beta), F32(lr), F32(eps)
    omb = F32(F32(1.0) - b)
    inv = None if grad_scale is None else F32(F32(1.0) / F32(grad_scale))
    for x in tensors:
        g = np.asarray(x.g).astype(F32)
        if inv is not None:
            g = g * inv
        wd = F32(x.wd)
        if wd > 0:
            g = g + x.p * wd
        if rule == "momentum":
            s = b * x.s + g
            d = s
        elif rule == "rmsprop":
            s = b * x.s + omb * (g * g)
            d = g / (np.sqrt(s) + eps32)
        else:
            s = x.s + g * g
            d = g / (np.sqrt(s) + eps32)
        x.p[...] = (x.p - lr32 * d).astype(F32)
        x.s[...] = s.astype(F32)
    return True
