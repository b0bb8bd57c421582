"""Pins for the AdEMAMix oracle (CPU only).

"Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
(bitsandbytes PR #2040): one step from a zero state reduces to the AdamW
closed form with alpha*(1-b3)*g mixed in, and the decay comes from the same
previous parameter as the update.  Further pins: alpha = 0 is AdamW (float64,
checked against the already pinned AdamW oracle and against torch's AdamW), the
slow EMA is not bias-corrected (b3 = 0 makes m2 = g exactly), strict-fp32 mode
tracks the float64 definition, and mutants fail.
"""

import numpy as np
import pytest
import torch

from oracle import ademamix as X
from oracle import adamw as A

f32 = A.f32
HP = dict(lr=f32(0.1), beta1=f32(0.9), beta2=f32(0.999), beta3=f32(0.9999), alpha=f32(5.0),
          eps=f32(1e-8))


def _state(n, seed, zero=True):
    rng = np.random.default_rng(seed)
    p = rng.normal(0, 0.02, n)
    g = rng.normal(0, 1e-3, n)
    z = [np.zeros(n) for _ in range(3)] if zero else [rng.normal(0, 1e-3, n), rng.normal(0, 1e-3, n),
                                                     rng.normal(0, 1e-3, n) ** 2]
    return p, g, z


def test_first_step_closed_form():
    p, g, (m1, m2, v) = _state(4096, 1)
    x = X.Tensor(p=p.copy(), g=g, m1=m1, m2=m2, v=v, wd=f32(0.1))
    X.step_fp64([x], t=1, **HP)
    lr, wd, eps, al, b3 = HP["lr"], f32(0.1), HP["eps"], HP["alpha"], HP["beta3"]
    want = p * (1 - lr * wd) - lr * (g + al * (1 - b3) * g) / (np.abs(g) + eps)
    assert np.allclose(x.p, want, rtol=1e-13, atol=1e-16)


def test_first_step_closed_form_f32():
    p, g, _ = _state(1 << 14, 2)
    p, g = p.astype(np.float32), g.astype(np.float32)
    z = [np.zeros_like(p) for _ in range(3)]
    x = X.Tensor(p=p.copy(), g=g, m1=z[0], m2=z[1], v=z[2], wd=f32(0.1))
    X.step_f32([x], t=1, **HP)
    lr, eps, al, b3 = np.float64(HP["lr"]), HP["eps"], HP["alpha"], HP["beta3"]
    pd, gd = p.astype(np.float64), g.astype(np.float64)
    want = pd * (1 - lr * f32(0.1)) - lr * (gd + al * (1 - b3) * gd) / (np.abs(gd) + eps)
    assert np.max(np.abs(x.p - want) / (np.abs(pd) + lr)) < 16 * 2.0 ** -24


def test_alpha_zero_is_adamw():
    p, g, (m1, m2, v) = _state(2048, 3, zero=False)
    hp = dict(HP, alpha=0.0)
    xs = X.Tensor(p=p.copy(), g=g, m1=m1.copy(), m2=m2.copy(), v=v.copy(), wd=0.05)
    ref = A.Tensor(p=p.copy(), g=g, m=m1.copy(), v=v.copy(), wd=0.05)
    for t in (1, 2, 3):
        X.step_fp64([xs], t=t, **hp)
        A.step_fp64([ref], lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"], t=t)
    assert np.max(np.abs(xs.p - ref.p)) < 1e-15
    assert np.array_equal(xs.m1, ref.m) and np.array_equal(xs.v, ref.v)


def test_alpha_zero_matches_torch_adamw():
    rng = np.random.default_rng(4)
    n = 1024
    p0 = rng.normal(0, 0.02, n)
    tp = torch.nn.Parameter(torch.tensor(p0))
    opt = torch.optim.AdamW([tp], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=f32(0.1), foreach=False)
    x = X.Tensor(p=p0.copy(), g=None, m1=np.zeros(n), m2=np.zeros(n), v=np.zeros(n), wd=f32(0.1))
    for t in range(1, 8):
        gr = rng.normal(0, 1e-3, n)
        tp.grad = torch.tensor(gr)
        opt.step()
        x.g = gr
        X.step_fp64([x], t=t, **dict(HP, alpha=0.0))
    assert np.max(np.abs(tp.detach().numpy() - x.p)) < 1e-13


def test_slow_ema_is_not_bias_corrected():
    p, g, (m1, m2, v) = _state(512, 5, zero=False)
    x = X.Tensor(p=p.copy(), g=g, m1=m1.copy(), m2=m2.copy(), v=v.copy(), wd=0.0)
    X.step_fp64([x], t=3, **dict(HP, beta3=0.0))
    assert np.array_equal(x.m2, g)


def test_decay_from_previous_parameter():
    p, g, (m1, m2, v) = _state(512, 6, zero=False)
    xs = [X.Tensor(p=p.copy(), g=g, m1=m1.copy(), m2=m2.copy(), v=v.copy(), wd=w) for w in (0.0, 0.2)]
    X.step_fp64(xs, t=2, **HP)
    assert np.allclose(xs[0].p - xs[1].p, p * HP["lr"] * 0.2, rtol=1e-12, atol=1e-15)


def test_f32_tracks_fp64_ten_steps():
    rng = np.random.default_rng(7)
    n = 1 << 15
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    x64 = X.Tensor(p=p0.astype(np.float64), g=None, m1=np.zeros(n), m2=np.zeros(n), v=np.zeros(n),
                   wd=f32(0.1))
    z = lambda: np.zeros(n, np.float32)
    x32 = X.Tensor(p=p0.copy(), g=None, m1=z(), m2=z(), v=z(), wd=f32(0.1))
    for t in range(1, 11):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        x64.g, x32.g = g.astype(np.float64), g
        X.step_fp64([x64], t=t, **HP)
        X.step_f32([x32], t=t, **HP)
    assert np.max(np.abs(x32.p - x64.p)) <= 5e-5 * 6     # alpha = 5 scales the update ~6x


@pytest.mark.parametrize("fn", [X.step_fp64, X.step_f32])
def test_skip(fn):
    dt = np.float64 if fn is X.step_fp64 else np.float32
    p, g, (m1, m2, v) = _state(300, 8, zero=False)
    p, g, m1, m2, v = (a.astype(dt) for a in (p, g * 128, m1, m2, v))
    g[17] = np.nan
    x = X.Tensor(p=p.copy(), g=g, m1=m1.copy(), m2=m2.copy(), v=v.copy(), wd=0.1)
    assert fn([x], t=2, grad_scale=128.0, **HP) is False
    assert np.array_equal(x.p, p) and np.array_equal(x.m2, m2)


def _mut_slow_bias_corrected(tensors, *, lr, beta1, beta2, beta3, alpha, eps, t, grad_scale=None):
    bc1, sqrt_bc2 = A.bias_corrections(beta1, beta2, t)
    bc3 = 1 - beta3 ** t
    for x in tensors:
        g = np.asarray(x.g, float)
        m1 = beta1 * x.m1 + (1 - beta1) * g
        m2 = beta3 * x.m2 + (1 - beta3) * g
        v = beta2 * x.v + (1 - beta2) * g * g
        u = (m1 / bc1 + alpha * m2 / bc3) / (np.sqrt(v) / sqrt_bc2 + eps)
        x.p[...] = x.p * (1 - lr * x.wd) - lr * u
        x.m1[...], x.m2[...], x.v[...] = m1, m2, v
    return True


def _mut_alpha_outside(tensors, *, lr, beta1, beta2, beta3, alpha, eps, t, grad_scale=None):
    bc1, sqrt_bc2 = A.bias_corrections(beta1, beta2, t)
    for x in tensors:
        g = np.asarray(x.g, float)
        m1 = beta1 * x.m1 + (1 - beta1) * g
        m2 = beta3 * x.m2 + (1 - beta3) * g
        v = beta2 * x.v + (1 - beta2) * g * g
        h = np.sqrt(v) / sqrt_bc2 + eps
        x.p[...] = x.p * (1 - lr * x.wd) - lr * (m1 / bc1 / h + alpha * m2)   # alpha*m2 not normalised
        x.m1[...], x.m2[...], x.v[...] = m1, m2, v
    return True


@pytest.mark.parametrize("mutant", [_mut_slow_bias_corrected, _mut_alpha_outside])
def test_closed_form_rejects_mutants(mutant):
    p, g, (m1, m2, v) = _state(4096, 1)
    x = X.Tensor(p=p.copy(), g=g, m1=m1, m2=m2, v=v, wd=f32(0.1))
    mutant([x], t=1, **HP)
    lr, wd, eps, al, b3 = HP["lr"], f32(0.1), HP["eps"], HP["alpha"], HP["beta3"]
    want = p * (1 - lr * wd) - lr * (g + al * (1 - b3) * g) / (np.abs(g) + eps)
    assert not np.allclose(x.p, want, rtol=1e-13, atol=1e-16)
