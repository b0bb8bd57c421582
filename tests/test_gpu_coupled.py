"""GPU parity: momentum SGD, RMSprop and Adagrad with coupled L2 decay
(adamw_coupled_step) against the oracle.

Bit-exact against the strict-fp32 oracle of the three rules on ragged tensor
lists (tensors with wd 0.1, 0 and -0.2; a non-positive wd adds nothing), in
the fp32 and bf16 + remainder modes and for fp32/fp16/bf16 grads, on 1-state
plans without exp_avg_sq and on tensors off the 16-byte grid (scalar path);
the AMP unscale and skip; a 2-state plan keeps its v untouched.
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import AdamWError, FusedAdamW
from oracle import adamw as A
from oracle import coupled as C
from oracle import remainder as R

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu
f32 = A.f32
SIZES = [1, 9, 2047, 2048, 2049, 8193, 30001, 0, 777]
WDS = [f32(0.1), 0.0, f32(-0.2)]
HP = {"momentum": dict(beta=f32(0.9), eps=0.0),
      "rmsprop": dict(beta=f32(0.99), eps=f32(1e-8)),
      "adagrad": dict(beta=0.0, eps=f32(1e-10))}


def _view(a, misalign):
    if not misalign:
        return dev(a)
    return dev(a, shift=1)   # one element off the 16-byte grid, guard bands on both sides


def _make(rule, mode, gdtype, seed, misalign=False):
    rng = np.random.default_rng(seed)
    dev_t, orc = [], []
    for i, n in enumerate(SIZES):
        s = rng.normal(0, 1e-3, n).astype(np.float32)
        if rule != "momentum":
            s = s * s
        wd = WDS[i % 3]
        if mode == "fp32":
            p = rng.normal(0, 0.02, n).astype(np.float32)
            d = dict(p=_view(p, misalign), r=None)
            master = p.copy()
        else:
            hi = (rng.normal(0, 0.02, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            rem = rng.integers(0, 1 << 15, n).astype(np.int16)
            d = dict(p=_view(hi.view(np.int16), misalign).view(torch.bfloat16), r=_view(rem, misalign))
            master = R.join(hi, rem)
        d.update(s=_view(s, misalign), g=empty(n, gdtype))
        dev_t.append(d)
        orc.append(C.Tensor(p=master, g=None, s=s.copy(), wd=wd))
    opt = FusedAdamW([d["p"] for d in dev_t], [d["g"] for d in dev_t], [d["s"] for d in dev_t],
                     None, [o.wd for o in orc], mode=mode,
                     param_rems=[d["r"] for d in dev_t] if mode == "bf16_rem" else None)
    return opt, dev_t, orc, rng


def _check(mode, dev_t, orc, tag):
    assert_guards_intact()
    for i, (d, o) in enumerate(zip(dev_t, orc)):
        if mode == "fp32":
            assert np.array_equal(host(d["p"]).view(np.uint32), o.p.view(np.uint32)), (tag, i, "p")
        else:
            hi, rem = R.split(o.p)
            assert np.array_equal(host(d["p"]).view(np.uint16), hi), (tag, i, "bf16")
            assert np.array_equal(host(d["r"]), rem), (tag, i, "rem")
        assert np.array_equal(host(d["s"]).view(np.uint32), o.s.view(np.uint32)), (tag, i, "s")


@pytest.mark.parametrize("rule", C.RULES)
@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
@pytest.mark.parametrize("gdtype", [torch.float32, torch.float16, torch.bfloat16])
def test_coupled_bitexact(rule, mode, gdtype):
    opt, dev_t, orc, rng = _make(rule, mode, gdtype, seed=61)
    lr, step = torch.tensor([f32(1e-2)], device="cuda"), zeros(1, torch.int32)
    for _ in range(4):
        for d, o in zip(dev_t, orc):
            x, wide = grads_of(rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32), gdtype)
            d["g"].copy_(x)
            o.g = wide
        opt.step_coupled(rule, lr, step, **HP[rule])
        C.step_f32(orc, rule=rule, lr=f32(1e-2), **HP[rule])
    torch.cuda.synchronize()
    _check(mode, dev_t, orc, rule)
    assert int(step.item()) == 4 and opt.status() == 0


@pytest.mark.parametrize("rule", C.RULES)
def test_coupled_scalar_path_on_misaligned_tensors(rule):
    opt, dev_t, orc, rng = _make(rule, "fp32", torch.float32, seed=62, misalign=True)
    lr, step = torch.tensor([f32(1e-2)], device="cuda"), zeros(1, torch.int32)
    for _ in range(2):
        for d, o in zip(dev_t, orc):
            x = rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32)
            d["g"].copy_(torch.from_numpy(x))
            o.g = x
        opt.step_coupled(rule, lr, step, **HP[rule])
        C.step_f32(orc, rule=rule, lr=f32(1e-2), **HP[rule])
    torch.cuda.synchronize()
    _check("fp32", dev_t, orc, "misaligned")


@pytest.mark.parametrize("rule", C.RULES)
def test_coupled_skip_and_unscale(rule):
    n = 20_000
    rng = np.random.default_rng(63)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    s0 = np.abs(rng.normal(0, 1e-3, n)).astype(np.float32)
    g0 = rng.normal(0, 1e-3, n).astype(np.float32)
    p, s, g = dev(p0), dev(s0), dev(g0 * 1000)
    opt = FusedAdamW([p], [g], [s], None, [f32(0.1)])
    lr, step = torch.tensor([f32(1e-2)], device="cuda"), zeros(1, torch.int32)
    scale, found = torch.tensor([1000.0], device="cuda"), zeros(1)
    g[3] = float("-inf")
    opt.check_nonfinite(found)
    opt.step_coupled(rule, lr, step, grad_scale=scale, found_inf=found, **HP[rule])
    torch.cuda.synchronize()
    assert int(step.item()) == 0 and np.array_equal(host(p), p0) and np.array_equal(host(s), s0)
    g.copy_(dev(g0 * 1000))
    opt.check_nonfinite(found)
    opt.step_coupled(rule, lr, step, grad_scale=scale, found_inf=found, **HP[rule])
    ref = C.Tensor(p=p0.copy(), g=(g0 * 1000).astype(np.float32), s=s0.copy(), wd=f32(0.1))
    assert C.step_f32([ref], rule=rule, lr=f32(1e-2), grad_scale=1000.0, **HP[rule])
    torch.cuda.synchronize()
    assert int(step.item()) == 1
    assert np.array_equal(host(p).view(np.uint32), ref.p.view(np.uint32))
    assert np.array_equal(host(s).view(np.uint32), ref.s.view(np.uint32))


def test_coupled_on_a_two_state_plan_leaves_v_alone_and_rejects_bad_rules():
    n = 5000
    rng = np.random.default_rng(64)
    p0, s0, v0, g0 = (np.abs(rng.normal(0, 1e-2, n)).astype(np.float32) for _ in range(4))
    p, s, v, g = dev(p0), dev(s0), dev(v0), dev(g0)
    opt = FusedAdamW([p], [g], [s], [v], [f32(0.1)])
    lr, step = torch.tensor([f32(1e-2)], device="cuda"), zeros(1, torch.int32)
    opt.step_coupled("rmsprop", lr, step, **HP["rmsprop"])
    ref = C.Tensor(p=p0.copy(), g=g0, s=s0.copy(), wd=f32(0.1))
    C.step_f32([ref], rule="rmsprop", lr=f32(1e-2), **HP["rmsprop"])
    torch.cuda.synchronize()
    assert np.array_equal(host(p).view(np.uint32), ref.p.view(np.uint32))
    assert np.array_equal(host(v), v0)
    with pytest.raises(AdamWError):
        from adamw_optimizer_step_tensor_gb300 import adamw_coupled_step
        adamw_coupled_step(opt.plan, 7, lr.data_ptr(), step.data_ptr(), 0.9, 1e-8, None, None, None)
    with pytest.raises(AdamWError):
        opt.step_coupled("momentum", lr, step, beta=1.0)
