"""Pins for the AdamW oracle (CPU only).

Each check ties ``oracle.adamw`` to something other than itself: the first-step
closed form and the decay-ordering gap law printed in "Fix decoupled weight
decay ordering in the CUDA Adam/AdEMAMix kernels" (bitsandbytes PR #2040),
torch's own CPU AdamW in float64 as an independent referee (the reviewer on
that page used it the same way and found decay-first identical to it), and
special cases.  ``test_pins_reject_mutants`` plants plausible mistakes in
copies of the oracle and shows that the pins fail on every one of them.
"""

import math

import numpy as np
import pytest
import torch

from oracle import adamw as A

f32 = A.f32


def _state(n, seed, zero_state=True):
    rng = np.random.default_rng(seed)
    p = rng.normal(0, 0.02, n)
    g = rng.normal(0, 1e-3, n)
    m = np.zeros(n) if zero_state else rng.normal(0, 1e-3, n)
    v = np.zeros(n) if zero_state else rng.normal(0, 1e-3, n) ** 2
    return p, g, m, v


def _fp64_step(p, g, m, v, wd, t, step_fn=A.step_fp64, **hp):
    x = A.Tensor(p=p.copy(), g=g, m=m.copy(), v=v.copy(), wd=wd)
    step_fn([x], t=t, **hp)
    return x


HP = dict(lr=f32(0.1), beta1=f32(0.9), beta2=f32(0.999), eps=f32(1e-8))


# ---------------------------------------------------------------- pin checks
def closed_form_holds(step_fn) -> bool:
    """First step from zero state: p1 = p0*(1 - lr*wd) - lr*g/(|g| + eps)."""
    p, g, m, v = _state(4096, 1)
    wd = f32(0.1)
    x = _fp64_step(p, g, m, v, wd, 1, step_fn, **HP)
    lr, eps = HP["lr"], HP["eps"]
    want = p * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    return bool(np.allclose(x.p, want, rtol=1e-13, atol=1e-16))


def torch_referee_holds(step_fn, lr=f32(1e-3), wd=f32(0.01), steps=20, seed=2) -> bool:
    """Multi-step agreement with torch.optim.AdamW (float64, CPU, single-tensor path)."""
    rng = np.random.default_rng(seed)
    n = 2048
    p0 = rng.normal(0, 0.02, n)
    grads = [rng.normal(0, 1e-3, n) for _ in range(steps)]
    tp = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([tp], lr=lr, betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=wd, foreach=False, fused=False)
    x = A.Tensor(p=p0.copy(), g=None, m=np.zeros(n), v=np.zeros(n), wd=wd)
    for t, gr in enumerate(grads, start=1):
        tp.grad = torch.tensor(gr, dtype=torch.float64)
        opt.step()
        x.g = gr
        step_fn([x], lr=lr, beta1=HP["beta1"], beta2=HP["beta2"], eps=HP["eps"], t=t)
    ref = tp.detach().numpy()
    # torch's moment update is a lerp, not b1*m + (1-b1)*g: same value, other
    # rounding; tens of float64 ulps after 10-20 steps at |p| < 1.  Any change
    # to the method moves p by at least ~lr*lr*wd >= 1e-8 here.
    return float(np.max(np.abs(ref - x.p))) <= 1e-13


def ordering_gap_holds(step_fn) -> bool:
    """decay-first vs decay-after differ after one step by lr*wd*|step_size*u| (~1.0e-3 at lr=wd=0.1)."""
    p, g, m, v = _state(4096, 3)
    wd = f32(0.1)
    first = _fp64_step(p, g, m, v, wd, 1, step_fn, **HP)
    after = _fp64_step(p, g, m, v, wd, 1, A.step_fp64, decay_after=True, **HP)
    lr, eps = HP["lr"], HP["eps"]
    ss_u = lr * g / (np.abs(g) + eps)          # step_size * u on the first step
    predicted = lr * wd * np.abs(ss_u)
    return bool(np.allclose(np.abs(first.p - after.p), predicted, rtol=1e-6, atol=1e-15))


PINS = [closed_form_holds, torch_referee_holds, ordering_gap_holds]


# ---------------------------------------------------------------- the pins
def test_first_step_closed_form():
    assert closed_form_holds(A.step_fp64)


def test_first_step_closed_form_f32():
    p, g, m, v = _state(1 << 14, 4)
    p, g, m, v = (a.astype(np.float32) for a in (p, g, m, v))
    wd = f32(0.1)
    x = A.Tensor(p=p.copy(), g=g, m=m.copy(), v=v.copy(), wd=wd)
    A.step_f32([x], t=1, **HP)
    lr, eps = np.float64(HP["lr"]), np.float64(HP["eps"])
    pd, gd = p.astype(np.float64), g.astype(np.float64)
    want = pd * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
    # a handful of float32 roundings on terms of size |p| and lr
    assert np.max(np.abs(x.p - want) / (np.abs(pd) + lr)) < 8 * 2.0 ** -24


def test_torch_fp64_referee():
    assert torch_referee_holds(A.step_fp64)
    assert torch_referee_holds(A.step_fp64, lr=f32(0.1), wd=f32(0.1), steps=10, seed=5)


def test_ordering_gap_one_step():
    assert ordering_gap_holds(A.step_fp64)
    # the page's number: at lr = wd = 0.1 the orderings are 1.0e-3 apart
    p, g, m, v = _state(4096, 3)
    first = _fp64_step(p, g, m, v, f32(0.1), 1, **HP)
    after = _fp64_step(p, g, m, v, f32(0.1), 1, decay_after=True, **HP)
    assert abs(np.max(np.abs(first.p - after.p)) - 1.0e-3) < 1e-6


def test_orderings_identical_at_wd0():
    p, g, m, v = _state(4096, 6, zero_state=False)
    for t in (1, 7):
        a = _fp64_step(p, g, m, v, 0.0, t, **HP)
        b = _fp64_step(p, g, m, v, 0.0, t, decay_after=True, **HP)
        assert np.array_equal(a.p, b.p)


def test_ordering_gap_grows_as_lr_squared():
    """20 steps at wd=0.01: the gap grows x100 per x10 in lr (page: 1.1e-9 ... 1.1e-3)."""
    rng = np.random.default_rng(8)
    n = 4096
    p0 = rng.normal(0, 0.02, n)
    grads = [rng.normal(0, 1e-3, n) for _ in range(20)]
    gaps = []
    for lr in (1e-4, 1e-3, 1e-2, 1e-1):
        runs = []
        for after in (False, True):
            x = A.Tensor(p=p0.copy(), g=None, m=np.zeros(n), v=np.zeros(n), wd=0.01)
            for t, gr in enumerate(grads, start=1):
                x.g = gr
                A.step_fp64([x], lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, t=t,
                            decay_after=after)
            runs.append(x.p)
        gaps.append(np.max(np.abs(runs[0] - runs[1])))
    ratios = [gaps[i + 1] / gaps[i] for i in range(3)]
    assert all(80 < r < 120 for r in ratios), (gaps, ratios)
    assert 1e-9 < gaps[0] < 1e-8 and 1e-4 < gaps[3] < 1e-2


def test_f32_mode_tracks_fp64_ten_steps():
    """Strict-fp32 vs float64 definition, 10 steps at lr = wd = 0.1: max |dp| <= 5e-5."""
    rng = np.random.default_rng(9)
    n = 1 << 16
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    x64 = A.Tensor(p=p0.astype(np.float64), g=None, m=np.zeros(n), v=np.zeros(n), wd=f32(0.1))
    x32 = A.Tensor(p=p0.copy(), g=None, m=np.zeros(n, np.float32), v=np.zeros(n, np.float32),
                   wd=f32(0.1))
    for t in range(1, 11):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        x64.g = g.astype(np.float64)
        x32.g = g
        A.step_fp64([x64], t=t, **HP)
        A.step_f32([x32], t=t, **HP)
    assert np.max(np.abs(x32.p - x64.p)) <= 5e-5


def test_f32_single_step_relative():
    """One strict-fp32 step from a non-zero state within 1e-6 of the definition,
    relative to the size of the terms that produce each output."""
    p, g, m, v = _state(1 << 15, 10, zero_state=False)
    p, g, m, v = (a.astype(np.float32) for a in (p, g, m, v))
    x32 = A.Tensor(p=p.copy(), g=g, m=m.copy(), v=v.copy(), wd=f32(0.1))
    x64 = A.Tensor(p=p.astype(np.float64), g=g.astype(np.float64), m=m.astype(np.float64),
                   v=v.astype(np.float64), wd=f32(0.1))
    A.step_f32([x32], t=3, **HP)
    A.step_fp64([x64], t=3, **HP)
    scale = np.maximum(np.abs(p), np.abs(x64.p)) + HP["lr"] * 10
    assert np.max(np.abs(x32.p - x64.p) / scale) < 1e-6
    for a32, a64, old in ((x32.m, x64.m, m), (x32.v, x64.v, v)):
        sc = np.maximum(np.abs(old), np.abs(a64)) + 1e-30
        assert np.max(np.abs(a32 - a64) / sc) < 1e-6


@pytest.mark.parametrize("bad", [math.inf, -math.inf, math.nan])
@pytest.mark.parametrize("fn", [A.step_fp64, A.step_f32])
def test_nonfinite_grad_skips_step(bad, fn):
    dt = np.float64 if fn is A.step_fp64 else np.float32
    p, g, m, v = (a.astype(dt) for a in _state(1000, 11, zero_state=False))
    xs = [A.Tensor(p=p.copy(), g=(g * 65536).copy(), m=m.copy(), v=v.copy(), wd=0.1)
          for _ in range(2)]
    xs[1].g[123] = bad
    assert fn(xs, t=4, grad_scale=65536.0, **HP) is False
    for x in xs:
        assert np.array_equal(x.p, p) and np.array_equal(x.m, m) and np.array_equal(x.v, v)


@pytest.mark.parametrize("fn", [A.step_fp64, A.step_f32])
def test_unscale_by_power_of_two_is_exact(fn):
    dt = np.float64 if fn is A.step_fp64 else np.float32
    p, g, m, v = (a.astype(dt) for a in _state(1000, 12, zero_state=False))
    a = A.Tensor(p=p.copy(), g=g * 65536, m=m.copy(), v=v.copy(), wd=0.1)
    b = A.Tensor(p=p.copy(), g=g.copy(), m=m.copy(), v=v.copy(), wd=0.1)
    fn([a], t=2, grad_scale=65536.0, **HP)
    fn([b], t=2, **HP)
    assert np.array_equal(a.p, b.p) and np.array_equal(a.m, b.m) and np.array_equal(a.v, b.v)


def test_no_skip_without_grad_scale():
    p, g, m, v = _state(10, 13)
    g[3] = math.inf
    x = A.Tensor(p=p.copy(), g=g, m=m.copy(), v=v.copy(), wd=0.1)
    assert A.step_fp64([x], t=1, **HP) is True
    assert not np.isfinite(x.p[3]) and np.isfinite(x.p[4])


def test_pow_binary_exact_small_and_accurate_large():
    from fractions import Fraction
    for b in (f32(0.9), f32(0.999), f32(0.95)):
        for t in (0, 1, 2, 3, 10, 100, 1000, 12345):
            exact = Fraction(b) ** t
            got = Fraction(A.pow_binary(b, t))
            if exact < Fraction(2) ** -1000:
                assert got == 0.0 or abs(got - exact) < Fraction(2) ** -1000   # underflow
            elif t <= 1:
                assert got == exact
            else:
                # each squaring doubles the relative error carried so far: <= t ulps
                assert abs(got - exact) <= exact * Fraction(t, 2 ** 52)


def test_bias_correction_closed_values():
    bc1, sbc2 = A.bias_corrections(0.5, 0.75, 2)
    assert bc1 == 0.75 and sbc2 == math.sqrt(1 - 0.5625)


def test_weight_decay_is_per_tensor():
    p, g, m, v = _state(512, 14)
    xs = [A.Tensor(p=p.copy(), g=g, m=m.copy(), v=v.copy(), wd=w) for w in (0.0, 0.1)]
    A.step_fp64(xs, t=1, **HP)
    lr = HP["lr"]
    assert np.allclose(xs[0].p - xs[1].p, p * lr * 0.1, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- mutation check
def _mut_eps_inside(tensors, *, lr, beta1, beta2, eps, t, grad_scale=None):
    bc1, sqrt_bc2 = A.bias_corrections(beta1, beta2, t)
    for x in tensors:
        g = np.asarray(x.g, float)
        m = beta1 * x.m + (1 - beta1) * g
        v = beta2 * x.v + (1 - beta2) * g * g
        u = m / ((np.sqrt(v) + eps) / sqrt_bc2)            # eps before the correction
        x.p[...] = x.p * (1 - lr * x.wd) - lr / bc1 * u
        x.m[...], x.v[...] = m, v
    return True


def _mut_no_bc1(tensors, *, lr, beta1, beta2, eps, t, grad_scale=None):
    bc1, sqrt_bc2 = A.bias_corrections(beta1, beta2, t)
    for x in tensors:
        g = np.asarray(x.g, float)
        m = beta1 * x.m + (1 - beta1) * g
        v = beta2 * x.v + (1 - beta2) * g * g
        u = m / (np.sqrt(v) / sqrt_bc2 + eps)
        x.p[...] = x.p * (1 - lr * x.wd) - lr * u            # bias correction of m dropped
        x.m[...], x.v[...] = m, v
    return True


def _mut_v_linear(tensors, *, lr, beta1, beta2, eps, t, grad_scale=None):
    bc1, sqrt_bc2 = A.bias_corrections(beta1, beta2, t)
    for x in tensors:
        g = np.asarray(x.g, float)
        m = beta1 * x.m + (1 - beta1) * g
        v = beta2 * x.v + (1 - beta2) * np.abs(g) * 1e-3   # g*g replaced
        u = m / (np.sqrt(v) / sqrt_bc2 + eps)
        x.p[...] = x.p * (1 - lr * x.wd) - lr / bc1 * u
        x.m[...], x.v[...] = m, v
    return True


def _mut_decay_lr_squared(tensors, *, lr, beta1, beta2, eps, t, grad_scale=None):
    bc1, sqrt_bc2 = A.bias_corrections(beta1, beta2, t)
    for x in tensors:
        g = np.asarray(x.g, float)
        m = beta1 * x.m + (1 - beta1) * g
        v = beta2 * x.v + (1 - beta2) * g * g
        u = m / (np.sqrt(v) / sqrt_bc2 + eps)
        x.p[...] = x.p * (1 - x.wd) - lr / bc1 * u           # decay not scaled by lr
        x.m[...], x.v[...] = m, v
    return True


def _mut_decay_after(tensors, **kw):
    return A.step_fp64(tensors, decay_after=True, **kw)


def _mut_beta_swap(tensors, *, lr, beta1, beta2, eps, t, grad_scale=None):
    return A.step_fp64(tensors, lr=lr, beta1=beta2, beta2=beta1, eps=eps, t=t)


@pytest.mark.parametrize("mutant", [_mut_eps_inside, _mut_no_bc1, _mut_v_linear,
                                    _mut_decay_lr_squared, _mut_decay_after, _mut_beta_swap])
def test_pins_reject_mutants(mutant):
    assert not all(pin(mutant) for pin in PINS)


def test_pins_accept_oracle():
    assert all(pin(A.step_fp64) for pin in PINS)


# ---------------------------------------------------------------- golden fixtures
def _golden(name):
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


@pytest.mark.parametrize("fn,dt", [(A.step_fp64, np.float64), (A.step_f32, np.float32)])
def test_golden_first_step_worked_by_hand(fn, dt):
    """Hand-worked first steps (eps = 0, all values binary fractions: exact in both modes)."""
    for c in _golden("first_step_worked.json")["cases"]:
        x = A.Tensor(p=np.array([c["p0"]], dt), g=np.array([c["g"]], dt),
                     m=np.zeros(1, dt), v=np.zeros(1, dt), wd=c["wd"])
        fn([x], lr=c["lr"], beta1=0.5, beta2=0.75, eps=c["eps"], t=1)
        assert x.p[0] == c["p1"], c


def test_golden_page_gap_figures():
    gold = _golden("bnb_pr2040_ordering.json")
    p, g, m, v = _state(4096, 3)
    first = _fp64_step(p, g, m, v, f32(0.1), 1, **HP)
    after = _fp64_step(p, g, m, v, f32(0.1), 1, decay_after=True, **HP)
    assert np.max(np.abs(first.p - after.p)) == pytest.approx(gold["one_step_gap_lr0.1_wd0.1"], rel=1e-3)
    fig = gold["gap_vs_lr_wd0.01_20_steps"]
    vals = [fig[k] for k in ("1e-4", "1e-3", "1e-2", "1e-1")]
    assert all(80 < vals[i + 1] / vals[i] < 120 for i in range(3))
