"""Pins for the Adam-mini oracle (CPU only).

"Adam-mini <> DTensor", ``AdamWMini`` listing: one second moment per block
(element, head or tensor) of ``mean(g*g)``; decay when wd > 0; the update
``lr * m * ((1/bc1) / h)``.  Pinned by what the method fixes, not by retyping
it:

* a block whose grads all have the same magnitude is indistinguishable from
  AdamW (every element's ``g*g`` equals the block mean), over several steps;
* block length 1 is AdamW itself (the listing's embedding branch);
* the first step from zero state is ``p*(1-lr*wd) - lr*g/(rms_b + eps)`` with
  ``rms_b`` the block's root mean square grad (bias corrections cancel);
* with eps = 0 the first step is invariant to scaling a block's grads, and
  permuting grads inside a block permutes its update;
* the mean is over the block (not the sum), wd <= 0 means no decay, the AMP
  skip leaves everything untouched;
* the strict-fp32 mode tracks float64 within a few float32 roundings.
"""

import numpy as np
import pytest

from oracle import adamw as A
from oracle import mini as M

F32 = np.float32
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _t(p, g, block, wd=0.1, m=None, v=None):
    n = p.size
    return M.Tensor(p=p.copy(), g=g, m=np.zeros(n) if m is None else m.copy(),
                    v=np.zeros(n // block) if v is None else v.copy(), wd=wd, block=block)


def test_equal_magnitude_blocks_are_adamw():
    rng = np.random.default_rng(1)
    n, block = 1024, 128
    p = rng.normal(0, 0.02, n)
    x = _t(p, None, block)
    y = A.Tensor(p=p.copy(), g=None, m=np.zeros(n), v=np.zeros(n), wd=0.1)
    for t in range(1, 6):
        mag = np.repeat(rng.uniform(1e-4, 1e-2, n // block), block)   # one magnitude per block
        g = mag * rng.choice([-1.0, 1.0], n)
        x.g, y.g = g, g
        M.step_fp64([x], t=t, **HP)
        A.step_fp64([y], t=t, **HP)
    assert np.allclose(x.p, y.p, rtol=1e-14, atol=1e-17)
    assert np.allclose(x.m, y.m, rtol=1e-14, atol=1e-20)
    assert np.allclose(np.repeat(x.v, block), y.v, rtol=1e-13, atol=1e-25)


def test_block_one_is_adamw_in_both_modes():
    rng = np.random.default_rng(2)
    n = 777
    p = rng.normal(0, 0.02, n)
    x = _t(p, None, 1)
    y = A.Tensor(p=p.copy(), g=None, m=np.zeros(n), v=np.zeros(n), wd=0.1)
    p32 = p.astype(F32)
    x32 = M.Tensor(p=p32.copy(), g=None, m=np.zeros(n, F32), v=np.zeros(n, F32), wd=A.f32(0.1), block=1)
    y32 = A.Tensor(p=p32.copy(), g=None, m=np.zeros(n, F32), v=np.zeros(n, F32), wd=A.f32(0.1))
    hp32 = dict(lr=A.f32(1e-3), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8))
    for t in range(1, 4):
        g = rng.normal(0, 1e-3, n)
        x.g, y.g = g, g
        M.step_fp64([x], t=t, **HP)
        A.step_fp64([y], t=t, **HP)
        x32.g = y32.g = g.astype(F32)
        M.step_f32([x32], t=t, **hp32)
        A.step_f32([y32], t=t, **hp32)
    assert np.allclose(x.p, y.p, rtol=1e-14, atol=1e-17)
    assert np.array_equal(x32.p, y32.p) and np.array_equal(x32.v, y32.v)


def test_first_step_closed_form():
    rng = np.random.default_rng(3)
    n, block = 4096, 256
    p = rng.normal(0, 0.02, n)
    g = rng.normal(0, 1e-3, n) * np.repeat(rng.uniform(0.1, 10, n // block), block)
    lr, wd, eps = 0.1, 0.1, 1e-8
    x = _t(p, g, block, wd=wd)
    M.step_fp64([x], lr=lr, beta1=0.9, beta2=0.999, eps=eps, t=1)
    rms = np.repeat(np.sqrt(np.mean(g.reshape(-1, block) ** 2, axis=1)), block)
    want = p * (1 - lr * wd) - lr * g / (rms + eps)
    assert np.allclose(x.p, want, rtol=1e-12, atol=1e-16)


def test_scale_invariance_and_permutation_with_zero_eps():
    rng = np.random.default_rng(4)
    n, block = 512, 64
    p = rng.normal(0, 0.02, n)
    g = rng.normal(0, 1e-3, n)
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=0.0, t=1)
    a = _t(p, g, block, wd=0.0)
    b = _t(p, g * 1000.0, block, wd=0.0)
    M.step_fp64([a], **hp)
    M.step_fp64([b], **hp)
    # compare the displacements (p may cancel against them); one rounding of p each
    assert np.allclose(a.p - p, b.p - p, rtol=1e-12, atol=1e-17)
    perm = np.concatenate([rng.permutation(block) + k * block for k in range(n // block)])
    c = _t(p[perm], g[perm], block, wd=0.0)
    M.step_fp64([c], **hp)
    assert np.allclose(c.p - p[perm], (a.p - p)[perm], rtol=1e-12, atol=1e-17)


def test_mean_not_sum():
    block = 8
    x = _t(np.zeros(block), np.array([1.0] + [0.0] * (block - 1)), block, wd=0.0)
    M.step_fp64([x], t=1, **HP)
    assert x.v[0] == pytest.approx((1 - 0.999) / block, rel=1e-15)


@pytest.mark.parametrize("fn,dt", [(M.step_fp64, np.float64), (M.step_f32, np.float32)])
def test_non_positive_wd_means_no_decay(fn, dt):
    rng = np.random.default_rng(5)
    p = rng.normal(0, 0.02, 256).astype(dt)
    g = rng.normal(0, 1e-3, 256).astype(dt)
    a = M.Tensor(p=p.copy(), g=g, m=np.zeros(256, dt), v=np.zeros(4, dt), wd=-0.5, block=64)
    b = M.Tensor(p=p.copy(), g=g, m=np.zeros(256, dt), v=np.zeros(4, dt), wd=0.0, block=64)
    fn([a], t=1, lr=A.f32(1e-3), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8))
    fn([b], t=1, lr=A.f32(1e-3), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8))
    assert np.array_equal(a.p, b.p)


@pytest.mark.parametrize("fn,dt", [(M.step_fp64, np.float64), (M.step_f32, np.float32)])
def test_skip(fn, dt):
    rng = np.random.default_rng(6)
    p = rng.normal(0, 0.02, 256).astype(dt)
    g = (rng.normal(0, 1e-3, 256) * 1024).astype(dt)
    g[9] = np.inf
    m0 = rng.normal(0, 1e-3, 256).astype(dt)
    v0 = np.full(2, 1e-6, dt)
    x = M.Tensor(p=p.copy(), g=g, m=m0.copy(), v=v0.copy(), wd=0.1, block=128)
    assert fn([x], t=3, grad_scale=1024.0, lr=0.1, beta1=0.9, beta2=0.999, eps=1e-8) is False
    assert np.array_equal(x.p, p) and np.array_equal(x.m, m0) and np.array_equal(x.v, v0)


def test_block_must_divide_numel():
    with pytest.raises(ValueError):
        M.step_fp64([_t(np.zeros(10), np.zeros(10), 4, v=np.zeros(2))], t=1, **HP)


def test_f32_tracks_fp64():
    rng = np.random.default_rng(7)
    blocks = [1, 64, 1024]
    xs64, xs32 = [], []
    for b in blocks:
        p = rng.normal(0, 0.02, 2048).astype(F32)
        xs64.append(M.Tensor(p=p.astype(np.float64), g=None, m=np.zeros(2048), v=np.zeros(2048 // b),
                             wd=A.f32(0.1), block=b))
        xs32.append(M.Tensor(p=p.copy(), g=None, m=np.zeros(2048, F32), v=np.zeros(2048 // b, F32),
                             wd=A.f32(0.1), block=b))
    hp = dict(lr=A.f32(1e-3), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8))
    for t in range(1, 4):
        for a, b in zip(xs64, xs32):
            g = rng.normal(0, 1e-3, 2048).astype(F32)
            a.g, b.g = g.astype(np.float64), g
        M.step_fp64(xs64, t=t, **hp)
        M.step_f32(xs32, t=t, **hp)
    for a, b in zip(xs64, xs32):
        assert np.max(np.abs(b.p - a.p) / (np.abs(a.p) + hp["lr"])) < 16 * 2.0 ** -24
        assert np.max(np.abs(b.v - a.v) / a.v) < 16 * 2.0 ** -24


def test_block_sum_in_pieces_equals_the_whole_block_mean():
    """Values on a 2^-12 grid below 4: every square and every partial sum is
    exact in float64, so any order of the block's sum gives the same S_b, and
    the mean summed over uneven pieces must equal block_mean_sq of the block."""
    rng = np.random.default_rng(41)
    n = 100_003
    g = (rng.integers(-4 * 4096, 4 * 4096, n) / 4096.0).astype(np.float32)
    cuts = [0, 17, 4096, 50_000, 50_001, 99_999, n]
    s = sum(M.block_sum_sq(g[a:b]) for a, b in zip(cuts[:-1], cuts[1:]))
    assert s == np.sum(g.astype(np.float64) ** 2)
    assert M.mean_from_sum(s, n) == M.block_mean_sq(g, n)[0]


def test_given_mean_follows_a_sample_of_the_block():
    """step_f32 on a sample of one block, with the block's mean given, equals the
    full step restricted to the sample, bit for bit (p, m, v)."""
    rng = np.random.default_rng(42)
    n = 40_000
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    m = rng.normal(0, 1e-3, n).astype(np.float32)
    v = np.array([1e-6], dtype=np.float32)
    idx = np.sort(rng.choice(n, 1000, replace=False))
    full = M.Tensor(p=p.copy(), g=g, m=m.copy(), v=v.copy(), wd=A.f32(0.1), block=n)
    part = M.Tensor(p=p[idx].copy(), g=g[idx], m=m[idx].copy(), v=v.copy(), wd=A.f32(0.1),
                    block=idx.size)
    hp = dict(lr=A.f32(1e-3), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8), t=3)
    M.step_f32([full], **hp)
    mean = M.mean_from_sum(M.block_sum_sq(g), n)
    M.step_f32([part], means=[np.array([mean])], **hp)
    assert np.array_equal(part.p.view(np.uint32), full.p[idx].view(np.uint32))
    assert np.array_equal(part.m.view(np.uint32), full.m[idx].view(np.uint32))
    assert np.array_equal(part.v.view(np.uint32), full.v.view(np.uint32))
    with pytest.raises(ValueError):
        M.step_f32([part], means=[np.array([mean])], grad_scale=A.f32(2.0), **hp)
