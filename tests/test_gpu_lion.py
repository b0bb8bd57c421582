"""GPU parity: the Lion step (adamw_lion_step) against the oracle.

Bit-exact against the strict-fp32 Lion oracle on ragged tensor lists, in the
fp32 and bf16 + remainder modes and for fp32/fp16/bf16 grads, on plans without
exp_avg_sq (the 1-state layout) and on tensors off the 16-byte grid (scalar
path).  Lion's own invariant is checked on the device output against inputs
only: after the decay every element moves by exactly lr, or not at all where
b1*m + (1-b1)*g is 0 ("Fix decoupled weight decay ordering in the CUDA
Adam/AdEMAMix kernels", bitsandbytes PR #2040: decay comes before the sign
update).  A plan that also carries v and a slow EMA leaves both untouched.
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import AdamWError, FusedAdamW
from oracle import adamw as A
from oracle import lion as L
from oracle import remainder as R

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu
f32 = A.f32
B1, B2 = f32(0.9), f32(0.99)
SIZES = [1, 9, 2047, 2048, 2049, 8193, 30001, 0, 777]


def _view(a, misalign):
    if not misalign:
        return dev(a)
    return dev(a, shift=1)   # one element off the 16-byte grid, guard bands on both sides


def _make(mode, gdtype, seed, misalign=False):
    rng = np.random.default_rng(seed)
    dev_t, orc = [], []
    for i, n in enumerate(SIZES):
        m = rng.normal(0, 1e-3, n).astype(np.float32)
        wd = f32(0.1) if i % 2 else 0.0
        if mode == "fp32":
            p = rng.normal(0, 0.02, n).astype(np.float32)
            d = dict(p=_view(p, misalign), r=None)
            master = p.copy()
        else:
            hi = (rng.normal(0, 0.02, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            rem = rng.integers(0, 1 << 15, n).astype(np.int16)
            d = dict(p=_view(hi.view(np.int16), misalign).view(torch.bfloat16), r=_view(rem, misalign))
            master = R.join(hi, rem)
        d.update(m=_view(m, misalign), g=empty(n, gdtype))
        dev_t.append(d)
        orc.append(L.Tensor(p=master, g=None, m=m.copy(), wd=wd))
    opt = FusedAdamW([d["p"] for d in dev_t], [d["g"] for d in dev_t], [d["m"] for d in dev_t],
                     None, [o.wd for o in orc], mode=mode,
                     param_rems=[d["r"] for d in dev_t] if mode == "bf16_rem" else None)
    return opt, dev_t, orc, rng


def _master(mode, d):
    if mode == "fp32":
        return host(d["p"])
    return R.join(host(d["p"]).view(np.uint16), host(d["r"]))


def _check(mode, dev_t, orc, tag):
    assert_guards_intact()
    for i, (d, o) in enumerate(zip(dev_t, orc)):
        if mode == "fp32":
            assert np.array_equal(host(d["p"]).view(np.uint32), o.p.view(np.uint32)), (tag, i, "p")
        else:
            hi, rem = R.split(o.p)
            assert np.array_equal(host(d["p"]).view(np.uint16), hi), (tag, i, "bf16")
            assert np.array_equal(host(d["r"]), rem), (tag, i, "rem")
        assert np.array_equal(host(d["m"]).view(np.uint32), o.m.view(np.uint32)), (tag, i, "m")


@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
@pytest.mark.parametrize("gdtype", [torch.float32, torch.float16, torch.bfloat16])
def test_lion_bitexact(mode, gdtype):
    opt, dev_t, orc, rng = _make(mode, gdtype, seed=51)
    lr, step = torch.tensor([f32(3e-4)], device="cuda"), zeros(1, torch.int32)
    for t in range(1, 5):
        for d, o in zip(dev_t, orc):
            x, wide = grads_of(rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32), gdtype)
            d["g"].copy_(x)
            o.g = wide
        opt.step_lion(lr, step, betas=(B1, B2))
        L.step_f32(orc, lr=f32(3e-4), beta1=B1, beta2=B2)
        torch.cuda.synchronize()
        _check(mode, dev_t, orc, t)
    assert int(step.item()) == 4 and opt.status() == 0


def test_lion_scalar_path_on_misaligned_tensors():
    opt, dev_t, orc, rng = _make("fp32", torch.float32, seed=52, misalign=True)
    lr, step = torch.tensor([f32(1e-3)], device="cuda"), zeros(1, torch.int32)
    for _ in range(2):
        for d, o in zip(dev_t, orc):
            x = rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32)
            d["g"].copy_(torch.from_numpy(x))
            o.g = x
        opt.step_lion(lr, step, betas=(B1, B2))
        L.step_f32(orc, lr=f32(1e-3), beta1=B1, beta2=B2)
    torch.cuda.synchronize()
    _check("fp32", dev_t, orc, "misaligned")


@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
def test_lion_moves_each_element_by_exactly_lr(mode):
    # checked from the inputs alone: p*fl(1 - lr*wd) is the one product the
    # kernel rounds before subtracting lr*sign, so |p' - p*decay| is lr up to
    # the rounding of that subtraction (half an ulp of the result)
    opt, dev_t, orc, rng = _make(mode, torch.float32, seed=53)
    lrv = f32(1e-3)
    lr, step = torch.tensor([lrv], device="cuda"), zeros(1, torch.int32)
    # exact zeros: m = g = 0 on a stretch of one tensor gives c = 0, so no move
    d6 = dev_t[6]
    d6["m"][100:200] = 0
    assert orc[6].wd == 0.0
    start6 = _master(mode, d6)[100:200].copy()
    for t in range(3):
        before = [_master(mode, d) for d in dev_t]
        ms = [host(d["m"]) for d in dev_t]
        gs = []
        for d in dev_t:
            x = rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32)
            if d is d6:
                x[100:200] = 0
            d["g"].copy_(torch.from_numpy(x))
            gs.append(x)
        opt.step_lion(lr, step, betas=(B1, B2))
        torch.cuda.synchronize()
        for d, o, p0, m0, g0 in zip(dev_t, orc, before, ms, gs):
            if p0.size == 0:
                continue
            decay = A.decay_f32(lrv, o.wd)
            c = np.float64(B1) * m0 + np.float64(1 - 0.9) * g0   # only its sign matters here
            moved = np.abs(_master(mode, d).astype(np.float64) - (p0 * decay).astype(np.float32).astype(np.float64))
            tol = (np.abs(p0).astype(np.float64) + lrv) * 2.0 ** -24
            want = np.where(np.abs(c) > 1e-12, np.float64(lrv), 0.0)
            assert np.all(np.abs(moved - want) <= tol), (mode, t)
    # c = 0 at every step there (m stays 0) and wd = 0: those elements never move
    assert np.array_equal(_master(mode, d6)[100:200].view(np.uint32), start6.view(np.uint32))


def test_lion_skip_and_unscale():
    n = 40_000
    rng = np.random.default_rng(54)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    m0 = rng.normal(0, 1e-3, n).astype(np.float32)
    g0 = rng.normal(0, 1e-3, n).astype(np.float32)
    p, m, g = dev(p0), dev(m0), dev(g0 * 128)
    opt = FusedAdamW([p], [g], [m], None, [f32(0.1)])
    lr, step = torch.tensor([f32(1e-3)], device="cuda"), zeros(1, torch.int32)
    scale, found = torch.tensor([128.0], device="cuda"), zeros(1)
    g[7] = float("nan")
    opt.check_nonfinite(found)
    opt.step_lion(lr, step, betas=(B1, B2), grad_scale=scale, found_inf=found)
    torch.cuda.synchronize()
    assert int(step.item()) == 0 and np.array_equal(host(p), p0) and np.array_equal(host(m), m0)
    g.copy_(dev(g0 * 128))
    opt.check_nonfinite(found)
    opt.step_lion(lr, step, betas=(B1, B2), grad_scale=scale, found_inf=found)
    ref = L.Tensor(p=p0.copy(), g=g0 * f32(128), m=m0.copy(), wd=f32(0.1))
    assert L.step_f32([ref], lr=f32(1e-3), beta1=B1, beta2=B2, grad_scale=128.0)
    torch.cuda.synchronize()
    assert int(step.item()) == 1
    assert np.array_equal(host(p).view(np.uint32), ref.p.view(np.uint32))
    assert np.array_equal(host(m).view(np.uint32), ref.m.view(np.uint32))


def test_lion_leaves_second_and_slow_states_alone():
    n = 10_000
    rng = np.random.default_rng(55)
    p0, m0, v0, s0, g0 = (rng.normal(0, 1e-2, n).astype(np.float32) for _ in range(5))
    p, m, v, s, g = dev(p0), dev(m0), dev(np.abs(v0)), dev(s0), dev(g0)
    opt = FusedAdamW([p], [g], [m], [v], [0.0], exp_avg_slows=[s])
    lr, step = torch.tensor([f32(1e-3)], device="cuda"), zeros(1, torch.int32)
    opt.step_lion(lr, step, betas=(B1, B2))
    ref = L.Tensor(p=p0.copy(), g=g0, m=m0.copy(), wd=0.0)
    L.step_f32([ref], lr=f32(1e-3), beta1=B1, beta2=B2)
    torch.cuda.synchronize()
    assert np.array_equal(host(p).view(np.uint32), ref.p.view(np.uint32))
    assert np.array_equal(host(v), np.abs(v0)) and np.array_equal(host(s), s0)


def test_one_state_plan_refuses_two_state_steps():
    n = 4096
    p, m, g = (zeros(n) for _ in range(3))
    opt = FusedAdamW([p], [g], [m], None, [0.0])
    lr, step = torch.tensor([f32(1e-3)], device="cuda"), zeros(1, torch.int32)
    with pytest.raises(AdamWError):
        opt.step(lr, step)
    found = zeros(1)
    with pytest.raises(AdamWError):
        opt.step_amp(lr, step, found)
    torch.cuda.synchronize()
    assert int(step.item()) == 0
