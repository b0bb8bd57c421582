"""Pins for the coupled-L2 1-state oracle (CPU only).

* torch.optim's SGD (momentum, no dampening), RMSprop and Adagrad in float64,
  with their own coupled ``weight_decay``, reach the same parameters over 20
  steps: an independent library routine for the exact same rules.
* Closed forms from zero state with a constant grad and no decay: momentum
  follows a geometric series, RMSprop's state is ``(1-b^k) g^2``, Adagrad's is
  ``k g^2`` ("Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix
  kernels", bitsandbytes PR #2040, names the three rules; their forms are the
  textbook ones).
* The decay goes into the grad (the page's coupled L2): the decoupled mutant
  is rejected, a non-positive wd adds nothing, and the decay term joins the
  grad after the unscale.
* The strict-fp32 mode agrees with float64 within a few float32 roundings.
"""

import numpy as np
import pytest

from oracle import adamw as A
from oracle import coupled as C

torch = pytest.importorskip("torch")


def _state(n, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(0, 0.5, n), rng.normal(0, 1e-2, n)


def _torch_opt(rule, params, lr, beta, eps, wd):
    if rule == "momentum":
        return torch.optim.SGD(params, lr=lr, momentum=beta, weight_decay=wd)
    if rule == "rmsprop":
        return torch.optim.RMSprop(params, lr=lr, alpha=beta, eps=eps, weight_decay=wd)
    return torch.optim.Adagrad(params, lr=lr, eps=eps, weight_decay=wd)


@pytest.mark.parametrize("rule", C.RULES)
def test_matches_torch_optim_float64(rule):
    p0, _ = _state(512, 1)
    lr, beta, eps, wd = 1e-2, 0.9, 1e-8, 0.1
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = _torch_opt(rule, [tp], lr, beta, eps, wd)
    x = C.Tensor(p=p0.copy(), g=None, s=np.zeros(512), wd=wd)
    rng = np.random.default_rng(7)
    for _ in range(20):
        g = rng.normal(0, 1e-2, 512)
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        x.g = g
        C.step_fp64([x], rule=rule, lr=lr, beta=beta, eps=eps)
    got = tp.detach().numpy()
    assert np.max(np.abs(got - x.p)) <= 1e-13 * (1 + np.max(np.abs(x.p)))


@pytest.mark.parametrize("rule", C.RULES)
def test_constant_grad_closed_forms(rule):
    g, p0, lr, b, eps, k = 3e-3, 0.25, 0.05, 0.8, 1e-8, 12
    x = C.Tensor(p=np.array([p0]), g=np.array([g]), s=np.zeros(1), wd=0.0)
    for _ in range(k):
        C.step_fp64([x], rule=rule, lr=lr, beta=b, eps=eps)
    j = np.arange(1, k + 1)
    if rule == "momentum":
        s_k = g * (1 - b ** k) / (1 - b)
        moves = g * (1 - b ** j) / (1 - b)
    elif rule == "rmsprop":
        s_k = (1 - b ** k) * g * g
        moves = g / (abs(g) * np.sqrt(1 - b ** j) + eps)
    else:
        s_k = k * g * g
        moves = g / (abs(g) * np.sqrt(j) + eps)
    assert x.s[0] == pytest.approx(s_k, rel=1e-13)
    assert x.p[0] == pytest.approx(p0 - lr * moves.sum(), rel=1e-13)


def test_momentum_zero_beta_is_plain_sgd_with_coupled_decay():
    p0, g = _state(64, 2)
    x = C.Tensor(p=p0.copy(), g=g, s=np.zeros(64), wd=0.5)
    C.step_fp64([x], rule="momentum", lr=0.1, beta=0.0)
    assert np.allclose(x.p, p0 - 0.1 * (g + 0.5 * p0), rtol=1e-15, atol=1e-17)
    assert np.allclose(x.s, g + 0.5 * p0, rtol=1e-15, atol=1e-17)


@pytest.mark.parametrize("rule", C.RULES)
def test_decoupled_mutant_differs(rule):
    p0, g = _state(256, 3)
    a = C.Tensor(p=p0.copy(), g=g, s=np.zeros(256), wd=0.1)
    b = C.Tensor(p=p0.copy(), g=g, s=np.zeros(256), wd=0.1)
    for _ in range(2):
        C.step_fp64([a], rule=rule, lr=0.1, beta=0.9, eps=1e-8)
        C.step_fp64([b], rule=rule, lr=0.1, beta=0.9, eps=1e-8, decoupled=True)
    assert np.max(np.abs(a.p - b.p)) > 1e-4


@pytest.mark.parametrize("rule", C.RULES)
@pytest.mark.parametrize("fn", [C.step_fp64, C.step_f32])
def test_non_positive_wd_adds_nothing(rule, fn):
    dt = np.float64 if fn is C.step_fp64 else np.float32
    p0, g = (a.astype(dt) for a in _state(128, 4))
    a = C.Tensor(p=p0.copy(), g=g, s=np.zeros(128, dt), wd=-0.3)
    b = C.Tensor(p=p0.copy(), g=g, s=np.zeros(128, dt), wd=0.0)
    fn([a], rule=rule, lr=1e-2, beta=0.9, eps=1e-8)
    fn([b], rule=rule, lr=1e-2, beta=0.9, eps=1e-8)
    assert np.array_equal(a.p, b.p) and np.array_equal(a.s, b.s)


@pytest.mark.parametrize("fn", [C.step_fp64, C.step_f32])
def test_decay_term_joins_the_unscaled_grad(fn):
    dt = np.float64 if fn is C.step_fp64 else np.float32
    p0, g = (a.astype(dt) for a in _state(128, 5))
    a = C.Tensor(p=p0.copy(), g=(g * 1024).astype(dt), s=np.zeros(128, dt), wd=0.25)
    b = C.Tensor(p=p0.copy(), g=g, s=np.zeros(128, dt), wd=0.25)
    assert fn([a], rule="momentum", lr=0.1, beta=0.9, grad_scale=1024.0)
    fn([b], rule="momentum", lr=0.1, beta=0.9)
    # a power-of-two scale unscales exactly, so the two must agree bit for bit
    assert np.array_equal(a.p, b.p) and np.array_equal(a.s, b.s)


@pytest.mark.parametrize("rule", C.RULES)
@pytest.mark.parametrize("fn", [C.step_fp64, C.step_f32])
def test_skip_on_nonfinite(rule, fn):
    dt = np.float64 if fn is C.step_fp64 else np.float32
    p0, g = (a.astype(dt) for a in _state(64, 6))
    g[3] = np.nan
    s0 = np.full(64, 0.5, dt)
    x = C.Tensor(p=p0.copy(), g=g, s=s0.copy(), wd=0.1)
    assert fn([x], rule=rule, lr=0.1, beta=0.9, eps=1e-8, grad_scale=8.0) is False
    assert np.array_equal(x.p, p0) and np.array_equal(x.s, s0)


@pytest.mark.parametrize("rule", C.RULES)
def test_f32_tracks_fp64(rule):
    p0, _ = _state(4096, 8)
    p32 = p0.astype(np.float32)
    x64 = C.Tensor(p=p32.astype(np.float64), g=None, s=np.zeros(4096), wd=A.f32(0.1))
    x32 = C.Tensor(p=p32.copy(), g=None, s=np.zeros(4096, np.float32), wd=A.f32(0.1))
    rng = np.random.default_rng(9)
    lr, b, eps = A.f32(1e-3), A.f32(0.9), A.f32(1e-8)
    for _ in range(3):
        g = rng.normal(0, 1e-2, 4096).astype(np.float32)
        x64.g, x32.g = g.astype(np.float64), g
        C.step_fp64([x64], rule=rule, lr=lr, beta=b, eps=eps)
        C.step_f32([x32], rule=rule, lr=lr, beta=b, eps=eps)
    # parameters of size ~0.5 moved by ~lr per step: the float32 roundings of p
    # dominate, a few ulps of |p|
    assert np.max(np.abs(x32.p - x64.p) / (np.abs(x64.p) + lr)) < 8 * 2.0 ** -24
    # the state sums terms that may cancel (g against p*wd): its error is a few
    # ulps of the largest state, not of each element
    assert np.max(np.abs(x32.s - x64.s)) / np.max(np.abs(x64.s)) < 64 * 2.0 ** -24
