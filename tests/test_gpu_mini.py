"""GPU parity: the Adam-mini step (adamw_mini_plan_create + adamw_mini_step).

Against the strict-fp32 Adam-mini oracle on ragged lists mixing block
lengths 1 (the AdamW branch), heads (several per tensor) and whole tensors,
with blocks that fit one chunk and blocks spread over many chunks (summed by
the last warp to arrive), in the fp32 and bf16 + remainder modes, for
fp32/fp16/bf16 grads.  The block means come from a float64 sum of exact
squares in the oracle and from error-free float32 pairs on the GPU: they agree
bit for bit except, rarely, by one ulp next to a rounding boundary, so v is
checked to one ulp (and nearly all bit-exact), m bit for bit, block-1 tensors
bit for bit, and the other parameters to the error one v ulp can cause.  One
step from zero state matches the closed form with the block RMS
(``p*(1-lr*wd) - lr*g/(rms + eps)``), and the AMP skip leaves everything alone.
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import AdamWError, FusedAdamW
from oracle import adamw as A
from oracle import mini as M
from oracle import remainder as R

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu
f32 = A.f32
HP = dict(beta1=f32(0.9), beta2=f32(0.999), eps=f32(1e-8))
# (numel, block): AdamW branch; heads in one chunk; one small tensor; odd whole
# tensor; heads over many chunks; a whole tensor over many chunks; empty
LAYOUT = [(50_000, 1), (64 * 12, 64), (2048, 2048), (777, 777), (3 * 40_000, 40_000),
          (100_003, 100_003), (16 * 300, 16), (0, 1)]
WDS = [f32(0.1), f32(0.1), 0.0, f32(0.1), f32(0.1), f32(-0.1), f32(0.1), 0.0]


def _make(mode, gdtype, seed):
    rng = np.random.default_rng(seed)
    dev_t, orc = [], []
    for (n, b), wd in zip(LAYOUT, WDS):
        m = rng.normal(0, 1e-3, n).astype(np.float32)
        v = (rng.normal(0, 1e-3, n // b) ** 2).astype(np.float32)
        if mode == "fp32":
            p = rng.normal(0, 0.02, n).astype(np.float32)
            d = dict(p=dev(p), r=None)
            master = p.copy()
        else:
            hi = (rng.normal(0, 0.02, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            rem = rng.integers(0, 1 << 15, n).astype(np.int16)
            d = dict(p=dev(hi.view(np.int16)).view(torch.bfloat16), r=dev(rem))
            master = R.join(hi, rem)
        d.update(m=dev(m), v=dev(v), g=empty(n, gdtype))
        dev_t.append(d)
        orc.append(M.Tensor(p=master, g=None, m=m.copy(), v=v.copy(), wd=wd, block=b))
    opt = FusedAdamW([d["p"] for d in dev_t], [d["g"] for d in dev_t], [d["m"] for d in dev_t],
                     [d["v"] for d in dev_t], [o.wd for o in orc], mode=mode,
                     param_rems=[d["r"] for d in dev_t] if mode == "bf16_rem" else None,
                     v_blocks=[b for _, b in LAYOUT])
    return opt, dev_t, orc, rng


def _master(mode, d):
    if mode == "fp32":
        return host(d["p"])
    return R.join(host(d["p"]).view(np.uint16), host(d["r"]))


def _ulps(a, b):
    ai = a.view(np.int32).astype(np.int64)
    bi = b.view(np.int32).astype(np.int64)
    return np.abs(ai - bi)


def _check(mode, dev_t, orc, lr, steps_done, tag):
    assert_guards_intact()
    exact_v = total_v = 0
    for i, (d, o) in enumerate(zip(dev_t, orc)):
        if o.p.size == 0:
            continue
        v = host(d["v"])
        u = _ulps(v, o.v)
        assert u.max() <= steps_done, (tag, i, "v", int(u.max()))
        exact_v += int(np.sum(u == 0))
        total_v += u.size
        assert np.array_equal(host(d["m"]).view(np.uint32), o.m.view(np.uint32)), (tag, i, "m")
        p = _master(mode, d)
        if o.block == 1:
            assert np.array_equal(p.view(np.uint32), o.p.view(np.uint32)), (tag, i, "p")
        else:
            # one v ulp moves r by about half an ulp: |dp| <= a few ulps of lr*|u|, plus p's rounding
            r_scale = np.abs(o.m).astype(np.float64) / np.sqrt(np.repeat(o.v, o.block).astype(np.float64) + 1e-30)
            tol = 2.0 ** -22 * (np.abs(o.p) + lr * r_scale * 4) * steps_done
            assert np.all(np.abs(p.astype(np.float64) - o.p) <= tol), (tag, i, "p")
    assert exact_v >= 0.98 * total_v, (tag, exact_v, total_v)


@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
@pytest.mark.parametrize("gdtype", [torch.float32, torch.float16, torch.bfloat16])
def test_mini_matches_oracle(mode, gdtype):
    opt, dev_t, orc, rng = _make(mode, gdtype, seed=71)
    lr_v = f32(1e-3)
    lr, step = torch.tensor([lr_v], device="cuda"), zeros(1, torch.int32)
    for t in range(1, 4):
        for d, o in zip(dev_t, orc):
            x, wide = grads_of(rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32), gdtype)
            d["g"].copy_(x)
            o.g = wide
        opt.step_mini(lr, step, betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"])
        M.step_f32(orc, lr=lr_v, t=t, **HP)
        torch.cuda.synchronize()
        _check(mode, dev_t, orc, lr_v, t, t)
    assert int(step.item()) == 3 and opt.status() == 0


def test_mini_reduction_is_deterministic():
    """Two copies of the same state and grads, stepped by two plans, agree bit
    for bit over three steps: the block sums are added in a fixed order, not in
    the order the warps of the reduction happen to arrive."""
    runs = []
    for _ in range(2):
        opt, dev_t, orc, rng = _make("fp32", torch.bfloat16, seed=75)
        lr, step = torch.tensor([f32(1e-3)], device="cuda"), zeros(1, torch.int32)
        for _t in range(3):
            for d in dev_t:
                x, _ = grads_of(rng.normal(0, 1e-3, d["g"].numel()).astype(np.float32),
                                torch.bfloat16)
                d["g"].copy_(x)
            opt.step_mini(lr, step, betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"])
        torch.cuda.synchronize()
        runs.append([{k: host(d[k]) for k in ("p", "m", "v")} for d in dev_t])
        del opt, dev_t
    for i, (a, b) in enumerate(zip(*runs)):
        for k in ("p", "m", "v"):
            assert bits_equal(a[k], b[k]), (i, k)


@pytest.mark.parametrize("gdtype", [torch.float16, torch.bfloat16, torch.float32])
def test_mini_with_a_loss_scale(gdtype):
    """The loss-scaled reduction and update (the scaled kernel instantiations):
    grads scaled by 3000 (not a power of two, so the unscale rounds), three
    steps, no non-finite grad -- against the oracle with the same scale."""
    opt, dev_t, orc, rng = _make("fp32", gdtype, seed=77)
    scale_v = 3000.0
    lr_v = f32(1e-3)
    lr, step = torch.tensor([lr_v], device="cuda"), zeros(1, torch.int32)
    scale = torch.tensor([scale_v], device="cuda")
    for t in range(1, 4):
        for d, o in zip(dev_t, orc):
            x, wide = grads_of((rng.normal(0, 1e-3, d["g"].numel()) * scale_v).astype(np.float32), gdtype)
            d["g"].copy_(x)
            o.g = wide
        opt.step_mini(lr, step, betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"], grad_scale=scale)
        assert M.step_f32(orc, lr=lr_v, t=t, grad_scale=f32(scale_v), **HP)
        torch.cuda.synchronize()
        _check("fp32", dev_t, orc, lr_v, t, t)
    assert int(step.item()) == 3 and opt.status() == 0


def test_mini_first_step_closed_form():
    rng = np.random.default_rng(72)
    n, block = 8 * 40_000, 40_000
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    g0 = (rng.normal(0, 1e-3, n) * np.repeat(rng.uniform(0.1, 10, n // block), block)).astype(np.float32)
    p, g = dev(p0), dev(g0)
    m, v = zeros(n), zeros(n // block)
    opt = FusedAdamW([p], [g], [m], [v], [f32(0.1)], v_blocks=[block])
    lr = f32(0.1)
    opt.step_mini(torch.tensor([lr], device="cuda"), zeros(1, torch.int32),
                  betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"])
    torch.cuda.synchronize()
    gd = g0.astype(np.float64)
    rms = np.repeat(np.sqrt(np.mean(gd.reshape(-1, block) ** 2, axis=1)), block)
    want = p0 * (1 - lr * f32(0.1)) - lr * gd / (rms + HP["eps"])
    got = host(p).astype(np.float64)
    assert np.max(np.abs(got - want) / (np.abs(want) + lr)) < 16 * 2.0 ** -24


def test_mini_skip_and_plan_rules():
    opt, dev_t, orc, rng = _make("fp32", torch.float16, seed=73)
    for d in dev_t:
        d["g"].copy_(dev((rng.normal(0, 1e-3, d["g"].numel()) * 1024).astype(np.float16)))
    dev_t[4]["g"][17] = float("inf")
    before = [{k: host(x) for k, x in d.items() if x is not None and k != "g"} for d in dev_t]
    found, step = zeros(1), zeros(1, torch.int32)
    scale = torch.tensor([1024.0], device="cuda")
    opt.check_nonfinite(found)
    opt.step_mini(torch.tensor([f32(1e-3)], device="cuda"), step, grad_scale=scale, found_inf=found)
    torch.cuda.synchronize()
    assert int(step.item()) == 0
    for d, b in zip(dev_t, before):
        for k, x in b.items():
            assert np.array_equal(host(d[k]).view(np.uint8), x.view(np.uint8)), k
    # a mini plan refuses the AdamW step (its v is per block)
    with pytest.raises(AdamWError):
        opt.step(torch.tensor([f32(1e-3)], device="cuda"), step)


def test_mini_llama_sized_blocks():
    """Blocks at Llama-3-8B sizes: 32 heads of 524,288 elements (one wq), one
    whole 58,720,256-element tensor (one w1), and a per-element tensor."""
    rng = np.random.default_rng(74)
    layout = [(32 * 524_288, 524_288), (14336 * 4096, 14336 * 4096), (4_000_000, 1)]
    ds, orc = [], []
    for n, b in layout:
        p = rng.normal(0, 0.02, n).astype(np.float32)
        g = rng.normal(0, 1e-4, n).astype(np.float32)
        ds.append(dict(p=dev(p), g=dev(g), m=zeros(n),
                       v=zeros(n // b)))
        orc.append(M.Tensor(p=p, g=g, m=np.zeros(n, np.float32), v=np.zeros(n // b, np.float32),
                            wd=f32(0.1), block=b))
    opt = FusedAdamW([d["p"] for d in ds], [d["g"] for d in ds], [d["m"] for d in ds],
                     [d["v"] for d in ds], [f32(0.1)] * 3, v_blocks=[b for _, b in layout])
    lr = f32(3e-4)
    opt.step_mini(torch.tensor([lr], device="cuda"), zeros(1, torch.int32),
                  betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"])
    M.step_f32(orc, lr=lr, t=1, **HP)
    torch.cuda.synchronize()
    _check("fp32", ds, orc, lr, 1, "llama-sized")
    del ds
    torch.cuda.empty_cache()


def test_mini_block_sums_past_the_float32_range():
    """Blocks of 256 whose squares or partial sums leave float32: one grad of
    1.9e19 (its square overflows, the block mean 1.4e36 does not), one +inf,
    one NaN, one -3e38 (the mean overflows too), and every grad 1e19 (the float32
    running sum overflows, the mean 1e38 does not) -- v as the float64 definition
    gives it: finite where the mean is, inf and NaN where they belong."""
    rng = np.random.default_rng(76)
    block = 256
    g0 = rng.normal(0, 1e-3, 6 * block).astype(np.float32)
    g0[3] = 1.9e19
    g0[block + 7] = np.inf
    g0[2 * block + 9] = np.nan
    g0[3 * block + 11] = -3e38
    g0[4 * block:5 * block] = 1e19
    n = g0.size
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    p, g, m, v = dev(p0), dev(g0), zeros(n), zeros(n // block)
    opt = FusedAdamW([p], [g], [m], [v], [f32(0.1)], v_blocks=[block])
    opt.step_mini(torch.tensor([f32(1e-3)], device="cuda"), zeros(1, torch.int32),
                  betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"])
    o = M.Tensor(p=p0.copy(), g=g0, m=np.zeros(n, np.float32), v=np.zeros(n // block, np.float32),
                 wd=f32(0.1), block=block)
    with np.errstate(invalid="ignore", over="ignore"):
        M.step_f32([o], lr=f32(1e-3), t=1, **HP)
    torch.cuda.synchronize()
    vd = host(v)
    assert np.isfinite(o.v[0]) and np.isfinite(o.v[4])        # the float64 means that stay finite
    assert np.isinf(o.v[1]) and np.isnan(o.v[2]) and np.isinf(o.v[3])
    assert np.array_equal(np.isnan(vd), np.isnan(o.v)) and np.array_equal(np.isinf(vd), np.isinf(o.v))
    fin = np.isfinite(o.v)
    assert np.all(_ulps(vd[fin], o.v[fin]) <= 1), (vd, o.v)
    assert opt.status() == 0
