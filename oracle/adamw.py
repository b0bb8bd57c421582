"""AdamW with decoupled weight decay -- CPU oracle (test infrastructure only).

Definition followed
-------------------
"Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
(bitsandbytes PR #2040), PR description: the decay and the gradient-based
update are both taken from the same previous parameter,
``p_new = p * (1 - lr*wd) + step_size * update``; the reviewer's torch.optim
excerpt on the same page shrinks the parameter before the moment updates.

"Adam-mini <> DTensor", the AdamW branch of the ``AdamWMini`` listing (the
embedding branch, which keeps full per-element ``v``): the moments
``m = b1*m + (1-b1)*g`` (written there as ``lerp``), ``v = b2*v + (1-b2)*g*g``,
``bc1 = 1 - b1**t``, ``bc2 = 1 - b2**t``, ``h = sqrt(v)/sqrt(bc2) + eps``,
``p += -(lr/bc1) * m / h``.  eps is added *after* the bias correction of
``sqrt(v)``; that is the only placement under which the first step from zero
state reduces to ``-lr * g / (|g| + eps)``, the closed form the bitsandbytes
PR description gives for its one-step 8-bit test.

"FusedAdam & PyTorch Lightning AMP", the maintainer's analysis: a fused step
receives the loss scale and a found-inf flag and does the unscale itself.
Reading taken here (the page does not spell the arithmetic out): grads are
divided by ``grad_scale``; if any raw grad of the step is inf or NaN the
whole step is skipped -- params, moments and the step counter are left
exactly as they were (GradScaler semantics: a skipped step is as if
``step()`` had not been called).

Two modes
---------
``step_fp64``  the definition, every value in float64.
``step_f32``   the *strict-fp32 specification*: the same sequence in float32,
               one IEEE round-to-nearest-even rounding per written operation,
               no fused multiply-add, in exactly the order written below.  The
               bias corrections are the one exception: ``b**t`` is taken by
               float64 binary exponentiation (``pow_binary``), ``1 - b**t``
               and ``1 / sqrt(1 - b2**t)`` in float64, each rounded to
               float32 once; the correction of ``sqrt(v)`` is applied as a
               multiplication by that reciprocal (the pages write a division
               and fix no rounding).  Discrete outputs (remainders, 8-bit
               codes) are defined against this mode.

Hyper-parameters are the float32 values the GPU entry point receives
(``lr`` read from a float32 device scalar; ``beta1``, ``beta2``, ``eps``,
``weight_decay`` and ``grad_scale`` as float32), promoted exactly to float64
in ``step_fp64``; pass float32-representable numbers (``f32(x)``) so both
modes see the same hyper-parameters.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

F32 = np.float32
F64 = np.float64


def f32(x: float) -> float:
    """Round a Python float to the nearest float32 and return it as a float."""
    return float(F32(x))


@dataclass
class Tensor:
    """One parameter tensor's state: param, grad, both moments, its weight decay.

    ``p``, ``m``, ``v`` are float arrays (float64 for ``step_fp64``, float32
    for ``step_f32``); ``g`` is the raw (possibly loss-scaled) gradient in any
    float dtype -- float16 and bfloat16-valued grads are passed already
    widened, which is exact.
    """

    p: np.ndarray
    g: np.ndarray
    m: np.ndarray
    v: np.ndarray
    wd: float


def pow_binary(b: float, t: int) -> float:
    """``b**t`` by float64 binary exponentiation (square-and-multiply).

    The exact operation sequence: ``r = 1; x = b; while t: if t & 1: r *= x;
    x *= x; t >>= 1``.  Every product is one float64 rounding, so any IEEE
    implementation of this loop yields the same bits.  Used instead of a
    library ``pow`` because a fast ``__powf`` was blamed for a 3e-6 error
    against the closed form in the bitsandbytes PR description.
    """
    if t < 0:
        raise ValueError("t must be >= 0")
    r = 1.0
    x = float(b)
    while t:
        if t & 1:
            r = r * x
        x = x * x
        t >>= 1
    return r


def bias_corrections(beta1: float, beta2: float, t: int) -> tuple[float, float]:
    """``(1 - beta1**t, sqrt(1 - beta2**t))`` in float64 (``pow_binary``)."""
    bc1 = 1.0 - pow_binary(beta1, t)
    bc2 = 1.0 - pow_binary(beta2, t)
    return bc1, math.sqrt(bc2)


def any_nonfinite(grads) -> bool:
    """True if any raw grad element of the step is +inf, -inf or NaN."""
    return any(not np.all(np.isfinite(np.asarray(g, dtype=F64))) for g in grads)


def step_fp64(tensors: list[Tensor], *, lr: float, beta1: float, beta2: float,
              eps: float, t: int, grad_scale: float | None = None,
              decay_after: bool = False) -> bool:
    """One AdamW step over a tensor list, in float64, in place.

    ``t`` is the 1-based index of this step (completed steps + 1).  Returns
    False (and changes nothing) when the step is skipped because a raw grad is
    non-finite and ``grad_scale`` is given (the AMP path); True otherwise.

    ``decay_after`` selects the *wrong* ordering the bitsandbytes PR removes,
    ``p = (p - step_size*u) * (1 - lr*wd)``.  It exists only so the tests can
    show they fail on it (the PR's own mutation check); the library has no
    such mode.
    """
    if grad_scale is not None and any_nonfinite([x.g for x in tensors]):
        return False
    b1, b2 = F64(beta1), F64(beta2)
    bc1, sqrt_bc2 = bias_corrections(beta1, beta2, t)
    step_size = F64(lr) / F64(bc1)
    for x in tensors:
        g = np.asarray(x.g, dtype=F64)
        if grad_scale is not None:
            g = g / F64(grad_scale)
        decay = F64(1.0) - F64(lr) * F64(x.wd)
        m = b1 * x.m + (F64(1.0) - b1) * g
        v = b2 * x.v + (F64(1.0) - b2) * g * g
        u = m / (np.sqrt(v) / F64(sqrt_bc2) + F64(eps))
        if decay_after:
            p = (x.p - step_size * u) * decay
        else:
            p = x.p * decay - step_size * u
        x.p[...] = p
        x.m[...] = m
        x.v[...] = v
    return True


@dataclass(frozen=True)
class F32Scalars:
    """Per-launch float32 scalars of the strict-fp32 specification."""

    b1: np.float32
    b2: np.float32
    omb1: np.float32      # fl(1 - b1)
    omb2: np.float32      # fl(1 - b2)
    eps: np.float32
    lr: np.float32
    step_size: np.float32  # fl(lr / bc1)
    inv_sqrt_bc2: np.float32   # fl32(1 / sqrt(1 - b2**t), both in float64)
    inv_scale: np.float32 | None  # fl(1 / grad_scale), None = no unscale
    sqrt_bc2: np.float32 = np.float32(1.0)   # fl32(sqrt(1 - b2**t)), for the division form


def f32_scalars(*, lr, beta1, beta2, eps, t, grad_scale=None) -> F32Scalars:
    """The launch-wide scalars, each rounded exactly as the specification says."""
    bc1, sqrt_bc2 = bias_corrections(float(F32(beta1)), float(F32(beta2)), t)
    b1, b2, lr32 = F32(beta1), F32(beta2), F32(lr)
    bc1_32 = F32(bc1)
    return F32Scalars(
        b1=b1, b2=b2, omb1=F32(F32(1.0) - b1), omb2=F32(F32(1.0) - b2),
        eps=F32(eps), lr=lr32, step_size=F32(lr32 / bc1_32),
        inv_sqrt_bc2=F32(1.0 / sqrt_bc2),
        inv_scale=None if grad_scale is None else F32(F32(1.0) / F32(grad_scale)),
        sqrt_bc2=F32(sqrt_bc2),
    )


def decay_f32(lr: np.float32, wd: float) -> np.float32:
    """Per-tensor decay factor ``fl(1 - fl(lr * wd))``."""
    return F32(F32(1.0) - F32(F32(lr) * F32(wd)))


def elementwise_f32(p, g_raw, m, v, s: F32Scalars, decay: np.float32, bias_rule="reciprocal",
                    decay_after=False):
    """The strict-fp32 element update; returns ``(p', m', v')`` as float32.

    Operation order (each line one rounding per operator, left to right):
        g   = g_raw                        (float32; fp16/bf16 widen exactly)
        g   = g * inv_scale                (only when a grad scale is given)
        m'  = b1*m + omb1*g
        v'  = b2*v + omb2*(g*g)
        h   = sqrt(v') * inv_sqrt_bc2 + eps
        u   = m' / h
        p'  = p*decay - step_size*u

    ``bias_rule="division"`` forms h as the AdamWMini listing of "Adam-mini <>
    DTensor" writes it, ``sqrt(v') / sqrt_bc2 + eps`` (one division per
    element); the library multiplies by the launch's ``inv_sqrt_bc2`` instead
    (the default here), a reading taken for speed.  The tests measure the
    distance between the two forms; nothing else uses the division form.

    ``decay_after`` is the *wrong* ordering the bitsandbytes PR removes,
    ``p' = (p - step_size*u) * decay``, in float32; it exists only so that the
    tests can show their GPU parity checks reject it (the PR's own mutation
    check).  The library has no such mode.
    """
    g = np.asarray(g_raw).astype(F32)
    if s.inv_scale is not None:
        g = g * s.inv_scale
    m1 = s.b1 * m + s.omb1 * g
    v1 = s.b2 * v + s.omb2 * (g * g)
    if bias_rule == "division":
        h = np.sqrt(v1) / s.sqrt_bc2 + s.eps
    else:
        h = np.sqrt(v1) * s.inv_sqrt_bc2 + s.eps
    u = m1 / h
    if decay_after:
        p1 = (p - s.step_size * u) * decay
    else:
        p1 = p * decay - s.step_size * u
    return p1.astype(F32), m1.astype(F32), v1.astype(F32)


def step_f32(tensors: list[Tensor], *, lr: float, beta1: float, beta2: float,
             eps: float, t: int, grad_scale: float | None = None) -> bool:
    """One AdamW step over a tensor list in the strict-fp32 specification, in place.

    Same contract as ``step_fp64``; ``p``, ``m``, ``v`` must be float32 arrays.
    """
    if grad_scale is not None and any_nonfinite([x.g for x in tensors]):
        return False
    s = f32_scalars(lr=lr, beta1=beta1, beta2=beta2, eps=eps, t=t,
                    grad_scale=grad_scale)
    for x in tensors:
        for a in (x.p, x.m, x.v):
            if a.dtype != F32:
                raise TypeError("step_f32 needs float32 p, m, v")
        p1, m1, v1 = elementwise_f32(x.p, x.g, x.m, x.v, s, decay_f32(s.lr, x.wd))
        x.p[...] = p1
        x.m[...] = m1
        x.v[...] = v1
    return True
