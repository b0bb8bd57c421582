"""Pins for the Lion oracle (CPU only).

The sign update makes every step's displacement exact: |p' - p*(1 - lr*wd)| is
lr (or 0 where the interpolation is exactly 0), at every step, not only the
first.  Decay comes first (bitsandbytes PR #2040 reviewer: Lion "applies
decoupled decay to the parameter before its sign update"), the direction uses
b1 while the state keeps the b2 EMA (a hand-made two-step case where the two
differ), and mutants fail.
"""

import numpy as np
import pytest

from oracle import adamw as A
from oracle import lion as L

f32 = A.f32


def _state(n, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(0, 0.02, n), rng.normal(0, 1e-3, n), rng.normal(0, 1e-3, n)


@pytest.mark.parametrize("fn,dt", [(L.step_fp64, np.float64), (L.step_f32, np.float32)])
def test_every_step_moves_by_exactly_lr(fn, dt):
    p, g, m = (a.astype(dt) for a in _state(4096, 1))
    lr, wd = f32(1e-3), f32(0.1)
    x = L.Tensor(p=p.copy(), g=g, m=m.copy(), wd=wd)
    for t in range(3):
        before = x.p.copy()
        x.g = (np.random.default_rng(t).normal(0, 1e-3, p.size)).astype(dt)
        c = dt(0.9) * x.m + (dt(1) - dt(0.9)) * x.g
        fn([x], lr=lr, beta1=0.9, beta2=0.99)
        decay = A.decay_f32(np.float32(lr), wd) if dt == np.float32 else 1 - lr * wd
        step = (before * dt(decay)).astype(np.float64) - x.p.astype(np.float64)
        # p*decay - lr*s rounds once (half an ulp of p'); the test's own p*decay is
        # the same rounded product, so the displacement is lr up to that rounding
        eps = 2.0 ** -53 if dt == np.float64 else 2.0 ** -24
        tol = eps * (np.abs(before).max() + lr) * 2
        assert np.all(np.abs(np.abs(step) - lr * (c != 0)) <= tol + 1e-18)


def test_decay_first_and_gap_to_decay_after():
    p, g, m = _state(2048, 2)
    lr, wd = 0.1, 0.1
    a = L.Tensor(p=p.copy(), g=g, m=m.copy(), wd=wd)
    b = L.Tensor(p=p.copy(), g=g, m=m.copy(), wd=wd)
    L.step_fp64([a], lr=lr, beta1=0.9, beta2=0.99)
    L.step_fp64([b], lr=lr, beta1=0.9, beta2=0.99, decay_after=True)
    assert np.allclose(np.abs(a.p - b.p), lr * wd * lr, rtol=1e-12)


def test_direction_uses_b1_state_uses_b2():
    x = L.Tensor(p=np.zeros(1), g=np.array([1.0]), m=np.zeros(1), wd=0.0)
    L.step_fp64([x], lr=1.0, beta1=0.9, beta2=0.99)
    assert x.p[0] == -1.0 and x.m[0] == pytest.approx(0.01)
    x.g = np.array([-0.2])
    # c = 0.9*0.01 + 0.1*(-0.2) = -0.011 < 0 (with b2 it would be +0.0079)
    L.step_fp64([x], lr=1.0, beta1=0.9, beta2=0.99)
    assert x.p[0] == 0.0
    assert x.m[0] == pytest.approx(0.99 * 0.01 + 0.01 * -0.2)


def test_sign_rules():
    c = np.array([0.0, -0.0, 1e-40, -1e-40, np.nan, np.inf, -3.0], np.float32)
    assert np.array_equal(L.sign(c), np.array([0, 0, 1, -1, 0, 1, -1], np.float32))


@pytest.mark.parametrize("fn", [L.step_fp64, L.step_f32])
def test_skip(fn):
    dt = np.float64 if fn is L.step_fp64 else np.float32
    p, g, m = (a.astype(dt) for a in _state(100, 3))
    g = g * 64
    g[5] = -np.inf
    x = L.Tensor(p=p.copy(), g=g, m=m.copy(), wd=0.1)
    assert fn([x], lr=1e-3, beta1=0.9, beta2=0.99, grad_scale=64.0) is False
    assert np.array_equal(x.p, p) and np.array_equal(x.m, m)


def test_f32_matches_fp64_where_direction_agrees():
    p, g, m = _state(1 << 14, 4)
    x64 = L.Tensor(p=p.astype(np.float32).astype(np.float64), g=g.astype(np.float32).astype(np.float64),
                   m=m.astype(np.float32).astype(np.float64), wd=f32(0.1))
    x32 = L.Tensor(p=p.astype(np.float32), g=g.astype(np.float32), m=m.astype(np.float32), wd=f32(0.1))
    L.step_fp64([x64], lr=f32(1e-3), beta1=f32(0.9), beta2=f32(0.99))
    L.step_f32([x32], lr=f32(1e-3), beta1=f32(0.9), beta2=f32(0.99))
    # same direction everywhere here; then p differs by float32 roundings only
    c64 = 0.9 * m.astype(np.float32).astype(np.float64) + 0.1 * g.astype(np.float32).astype(np.float64)
    assert np.all(np.abs(c64) > 1e-9)
    assert np.max(np.abs(x32.p - x64.p) / (np.abs(x64.p) + 1e-3)) < 4 * 2.0 ** -24
    # relative to the size of the terms of b2*m + (1-b2)*g (they may cancel)
    mm, gg = m.astype(np.float32).astype(np.float64), g.astype(np.float32).astype(np.float64)
    terms = 0.99 * np.abs(mm) + 0.01 * np.abs(gg)
    assert np.max(np.abs(x32.m - x64.m) / terms) < 4 * 2.0 ** -24
