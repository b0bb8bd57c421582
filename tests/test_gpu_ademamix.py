"""GPU parity: the AdEMAMix step (adamw_ademamix_step) against the oracle.

Bit-exact against the strict-fp32 AdEMAMix oracle on ragged tensor lists, in
the fp32 and bf16 + remainder modes and for fp32/fp16/bf16 grads (also on
tensors off the 16-byte grid, which take the scalar path); one step from zero
state follows the closed form of "Fix decoupled weight decay ordering in the
CUDA Adam/AdEMAMix kernels" (bitsandbytes PR #2040) with alpha*(1-b3)*g mixed in.
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW
from oracle import ademamix as X
from oracle import adamw as A
from oracle import remainder as R

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu
f32 = A.f32
HP = dict(beta1=f32(0.9), beta2=f32(0.999), beta3=f32(0.9999), alpha=f32(5.0), eps=f32(1e-8))
SIZES = [1, 9, 2047, 2048, 2049, 8193, 30001, 0, 777]


def _view(a, misalign):
    if not misalign:
        return dev(a)
    return dev(a, shift=1)   # one element off the 16-byte grid, guard bands on both sides


def _make(mode, gdtype, seed, misalign=False):
    rng = np.random.default_rng(seed)
    dev_t, orc = [], []
    for i, n in enumerate(SIZES):
        m1 = rng.normal(0, 1e-3, n).astype(np.float32)
        m2 = rng.normal(0, 1e-3, n).astype(np.float32)
        v = (rng.normal(0, 1e-3, n) ** 2).astype(np.float32)
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
        d.update(m=_view(m1, misalign), m2=_view(m2, misalign), v=_view(v, misalign),
                 g=empty(n, gdtype))
        dev_t.append(d)
        orc.append(X.Tensor(p=master, g=None, m1=m1.copy(), m2=m2.copy(), v=v.copy(), wd=wd))
    opt = FusedAdamW([d["p"] for d in dev_t], [d["g"] for d in dev_t], [d["m"] for d in dev_t],
                     [d["v"] for d in dev_t], [o.wd for o in orc], mode=mode,
                     param_rems=[d["r"] for d in dev_t] if mode == "bf16_rem" else None,
                     exp_avg_slows=[d["m2"] for d in dev_t])
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
        for k, ref in (("m", o.m1), ("m2", o.m2), ("v", o.v)):
            assert np.array_equal(host(d[k]).view(np.uint32), ref.view(np.uint32)), (tag, i, k)


@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
@pytest.mark.parametrize("gdtype", [torch.float32, torch.float16, torch.bfloat16])
def test_ademamix_bitexact(mode, gdtype):
    opt, dev_t, orc, rng = _make(mode, gdtype, seed=41)
    lr, step = torch.tensor([f32(3e-3)], device="cuda"), zeros(1, torch.int32)
    for t in range(1, 5):
        for d, o in zip(dev_t, orc):
            x, wide = grads_of(rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32), gdtype)
            d["g"].copy_(x)
            o.g = wide
        opt.step_ademamix(lr, step, betas=(HP["beta1"], HP["beta2"], HP["beta3"]), alpha=HP["alpha"],
                          eps=HP["eps"])
        X.step_f32(orc, lr=f32(3e-3), t=t, **HP)
        torch.cuda.synchronize()
        _check(mode, dev_t, orc, t)
    assert int(step.item()) == 4 and opt.status() == 0


def test_ademamix_scalar_path_on_misaligned_tensors():
    opt, dev_t, orc, rng = _make("fp32", torch.float32, seed=42, misalign=True)
    lr, step = torch.tensor([f32(1e-3)], device="cuda"), zeros(1, torch.int32)
    for t in (1, 2):
        for d, o in zip(dev_t, orc):
            x = rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32)
            d["g"].copy_(torch.from_numpy(x))
            o.g = x
        opt.step_ademamix(lr, step, betas=(HP["beta1"], HP["beta2"], HP["beta3"]), alpha=HP["alpha"],
                          eps=HP["eps"])
        X.step_f32(orc, lr=f32(1e-3), t=t, **HP)
    torch.cuda.synchronize()
    _check("fp32", dev_t, orc, "misaligned")


def test_ademamix_first_step_closed_form_and_skip():
    n = 50_000
    rng = np.random.default_rng(43)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    g0 = rng.normal(0, 1e-3, n).astype(np.float32)
    p = dev(p0)
    g = dev(g0 * 64)
    z = [zeros(n) for _ in range(3)]
    opt = FusedAdamW([p], [g], [z[0]], [z[1]], [f32(0.1)], exp_avg_slows=[z[2]])
    lr, step = torch.tensor([f32(0.1)], device="cuda"), zeros(1, torch.int32)
    scale, found = torch.tensor([64.0], device="cuda"), zeros(1)
    # a skipped step first: nothing moves
    g[11] = float("inf")
    opt.check_nonfinite(found)
    opt.step_ademamix(lr, step, betas=(HP["beta1"], HP["beta2"], HP["beta3"]), alpha=HP["alpha"],
                      eps=HP["eps"], grad_scale=scale, found_inf=found)
    torch.cuda.synchronize()
    assert int(step.item()) == 0 and np.array_equal(host(p), p0)
    g.copy_(dev(g0 * 64))
    opt.check_nonfinite(found)
    opt.step_ademamix(lr, step, betas=(HP["beta1"], HP["beta2"], HP["beta3"]), alpha=HP["alpha"],
                      eps=HP["eps"], grad_scale=scale, found_inf=found)
    torch.cuda.synchronize()
    lrd, al, b3, eps = np.float64(f32(0.1)), HP["alpha"], HP["beta3"], HP["eps"]
    pd, gd = p0.astype(np.float64), g0.astype(np.float64)
    want = pd * (1 - lrd * f32(0.1)) - lrd * (gd + al * (1 - b3) * gd) / (np.abs(gd) + eps)
    got = host(p).astype(np.float64)
    assert int(step.item()) == 1
    assert np.max(np.abs(got - want) / (np.abs(pd) + lrd)) < 16 * 2.0 ** -24
