"""GPU parity on the method's degenerate inputs, in the fp32 and bf16 + remainder
modes, on both the small-plan kernel and the bulk kernel.

Cases: special grads (NaN, +-inf, +-0, the smallest subnormals, grads whose
square overflows float32) reaching the update without a loss-scale skip;
lr = 0; beta1 = beta2 = 0 (bias corrections of exactly 1); eps = 0 on a zero
state with zero grads (0/0); a negative weight decay.  Every finite result must
equal the strict-fp32 oracle bit for bit.  A NaN result must be a NaN on both
sides: IEEE fixes that the result is a NaN, not its bits, and GPU arithmetic
returns its own NaN pattern where numpy keeps an input's payload.  In bf16 +
remainder mode the stored pair is compared bit for bit everywhere, NaNs
included, because the split stores every NaN master as the quiet NaN -- so a
NaN parameter is a NaN in the bf16 model weights, never a -0.0.
"""

import zlib

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW
from oracle import adamw as OA
from oracle import remainder as OR

from _support import assert_guards_intact, dev, empty, grads_of, host, scalar_f32, scalar_i32

pytestmark = pytest.mark.gpu
f32 = OA.f32

# the special grads, written at the front of every tensor and scattered in it
SPECIAL = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0, 1e-45, -1e-45, 3e38, -3e38,
                    1e-20, -1e-20, 1.5e19], dtype=np.float32)
SMALL = [64, 1000, 4099]                 # a small plan: one launch of the small kernel
BULK = [2048 + 37 * i for i in range(20)]  # 20 tensors: the bulk kernel

CASES = {
    "special_grads": dict(lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.1),
    "lr_zero": dict(lr=0.0, b1=0.9, b2=0.999, eps=1e-8, wd=0.1),
    "betas_zero": dict(lr=1e-3, b1=0.0, b2=0.0, eps=1e-8, wd=0.1),
    "eps_zero_on_zero_state": dict(lr=1e-3, b1=0.9, b2=0.999, eps=0.0, wd=0.1, zero_state=True),
    "negative_wd": dict(lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=-0.1),
}


def _grads(n, rng, zero_state):
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    k = min(n, SPECIAL.size)
    g[:k] = SPECIAL[:k]
    pos = rng.integers(0, n, 8)
    g[pos] = SPECIAL[rng.integers(0, SPECIAL.size, 8)]
    if zero_state:
        g[rng.integers(0, n, 16)] = 0.0      # 0/0 there once eps is 0
    return g


def _same_or_both_nan(a, b):
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


def _build(mode, sizes, gdtype, case, rng):
    import synth
    from _support import to_dev
    dev_t, orc = [], []
    for i, n in enumerate(sizes):
        if case.get("zero_state"):
            m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
        else:
            m = rng.normal(0, 1e-3, n).astype(np.float32)
            v = (rng.normal(0, 1e-3, n) ** 2).astype(np.float32)
        if mode == "fp32":
            p = rng.normal(0, 0.02, n).astype(np.float32)
            d = dict(p=dev(p), r=None)
            master = p.copy()
        else:
            hi, rem = synth.bf16_params_with_remainders(n, 0.02, seed=500 + i, device="cpu", n_zeros=8)
            d = dict(p=to_dev(hi), r=to_dev(rem))
            master = OR.join(hi.view(torch.int16).numpy().view(np.uint16), rem.numpy())
        d.update(m=dev(m), v=dev(v), g=empty(n, gdtype))
        dev_t.append(d)
        orc.append(OA.Tensor(p=master, g=None, m=m.copy(), v=v.copy(), wd=f32(case["wd"])))
    opt = FusedAdamW([d["p"] for d in dev_t], [d["g"] for d in dev_t], [d["m"] for d in dev_t],
                     [d["v"] for d in dev_t], [f32(case["wd"])] * len(sizes), mode=mode,
                     param_rems=[d["r"] for d in dev_t] if mode == "bf16_rem" else None)
    return opt, dev_t, orc


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("kernel", ["small", "bulk"])
@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
@pytest.mark.parametrize("gdtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_degenerate_inputs_match_the_oracle(case, kernel, mode, gdtype):
    c = CASES[case]
    rng = np.random.default_rng(zlib.crc32(f"{case}/{kernel}/{mode}/{gdtype}".encode()))
    sizes = SMALL if kernel == "small" else BULK
    opt, dev_t, orc = _build(mode, sizes, gdtype, c, rng)
    assert opt.info()["block_threads"] == (1024 if kernel == "small" else 544)
    hp = dict(beta1=f32(c["b1"]), beta2=f32(c["b2"]), eps=f32(c["eps"]))
    lr, step = scalar_f32(f32(c["lr"])), scalar_i32(0)
    for t in (1, 2):
        for d, o, n in zip(dev_t, orc, sizes):
            x, wide = grads_of(_grads(n, rng, c.get("zero_state", False)), gdtype)
            d["g"].copy_(x)
            o.g = wide
        opt.step(lr, step, betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"])
        with np.errstate(invalid="ignore", over="ignore", divide="ignore"):   # NaN / inf by design
            OA.step_f32(orc, lr=f32(c["lr"]), t=t, **hp)
    torch.cuda.synchronize()
    assert_guards_intact()
    n_nan = 0
    for i, (d, o) in enumerate(zip(dev_t, orc)):
        assert _same_or_both_nan(host(d["m"]), o.m), (i, "m")
        assert _same_or_both_nan(host(d["v"]), o.v), (i, "v")
        n_nan += int(np.isnan(o.p).sum())
        if mode == "fp32":
            assert _same_or_both_nan(host(d["p"]), o.p), (i, "p")
        else:
            ohi, orem = OR.split(o.p)
            hi = host(d["p"].view(torch.int16)).view(np.uint16)
            assert np.array_equal(hi, ohi), (i, "bf16 half")
            assert np.array_equal(host(d["r"]), orem), (i, "remainder")
            # a NaN parameter is a NaN in the model's bf16 weights
            assert np.all(np.isnan(OR.bf16_bits_to_f32(hi)[np.isnan(o.p)])), (i, "NaN -> bf16")
    assert int(step.item()) == 2 and opt.status() == 0
    if case in ("special_grads", "eps_zero_on_zero_state"):
        assert n_nan > 0      # the case reached the non-finite results it is about
    opt.close()


RULE_SIZES = [4096, 8192, 2048, 1000]
MINI_BLOCKS = [1, 8192, 256, 1]        # per element, one v per tensor, per 256-element head


def _rule_setup(rule, mode, rng):
    """The plan, the device tensors, the oracle tensors and the two step callables
    of one rule; the state names are the device keys after "p"."""
    import synth
    from oracle import ademamix as AD
    from oracle import coupled as CP
    from oracle import lion as LI
    from oracle import mini as MI
    from _support import to_dev
    wd = f32(0.1)
    dev_t, orc = [], []
    for i, n in enumerate(RULE_SIZES):
        if mode == "fp32":
            p = rng.normal(0, 0.02, n).astype(np.float32)
            d = dict(p=dev(p), r=None)
            master = p.copy()
        else:
            hi, rem = synth.bf16_params_with_remainders(n, 0.02, seed=600 + i, device="cpu", n_zeros=8)
            d = dict(p=to_dev(hi), r=to_dev(rem))
            master = OR.join(hi.view(torch.int16).numpy().view(np.uint16), rem.numpy())
        m = rng.normal(0, 1e-3, n).astype(np.float32)
        sq = (rng.normal(0, 1e-3, n) ** 2).astype(np.float32)
        d.update(g=empty(n, torch.float32), m=dev(m))
        if rule == "ademamix":
            m2 = rng.normal(0, 1e-3, n).astype(np.float32)
            d.update(m2=dev(m2), v=dev(sq))
            orc.append(AD.Tensor(p=master, g=None, m1=m.copy(), m2=m2.copy(), v=sq.copy(), wd=wd))
        elif rule == "lion":
            orc.append(LI.Tensor(p=master, g=None, m=m.copy(), wd=wd))
        elif rule == "mini":
            v = sq[: n // MINI_BLOCKS[i]].copy()
            d.update(v=dev(v))
            orc.append(MI.Tensor(p=master, g=None, m=m.copy(), v=v.copy(), wd=wd, block=MINI_BLOCKS[i]))
        else:
            s0 = m if rule == "momentum" else sq
            d["m"] = dev(s0)
            orc.append(CP.Tensor(p=master, g=None, s=s0.copy(), wd=wd))
        dev_t.append(d)
    rems = [d["r"] for d in dev_t] if mode == "bf16_rem" else None
    ps, gs, ms = [d["p"] for d in dev_t], [d["g"] for d in dev_t], [d["m"] for d in dev_t]
    kw = dict(mode=mode, param_rems=rems)
    if rule == "ademamix":
        opt = FusedAdamW(ps, gs, ms, [d["v"] for d in dev_t], [wd] * 4,
                         exp_avg_slows=[d["m2"] for d in dev_t], **kw)
        hp = dict(beta1=f32(0.9), beta2=f32(0.999), beta3=f32(0.9999), alpha=f32(5.0), eps=f32(1e-8))
        run = lambda lr, st: opt.step_ademamix(lr, st, betas=(hp["beta1"], hp["beta2"], hp["beta3"]),
                                               alpha=hp["alpha"], eps=hp["eps"])
        ref = lambda lr, t: AD.step_f32(orc, lr=lr, t=t, **hp)
        keys = (("m", "m1"), ("m2", "m2"), ("v", "v"))
    elif rule == "lion":
        opt = FusedAdamW(ps, gs, ms, None, [wd] * 4, **kw)
        run = lambda lr, st: opt.step_lion(lr, st, betas=(f32(0.9), f32(0.99)))
        ref = lambda lr, t: LI.step_f32(orc, lr=lr, beta1=f32(0.9), beta2=f32(0.99))
        keys = (("m", "m"),)
    elif rule == "mini":
        opt = FusedAdamW(ps, gs, ms, [d["v"] for d in dev_t], [wd] * 4, v_blocks=MINI_BLOCKS, **kw)
        run = lambda lr, st: opt.step_mini(lr, st, betas=(f32(0.9), f32(0.999)), eps=f32(1e-8))
        ref = lambda lr, t: MI.step_f32(orc, lr=lr, beta1=f32(0.9), beta2=f32(0.999), eps=f32(1e-8), t=t)
        keys = (("m", "m"), ("v", "v"))
    else:
        opt = FusedAdamW(ps, gs, ms, None, [wd] * 4, **kw)
        run = lambda lr, st: opt.step_coupled(rule, lr, st, beta=f32(0.9), eps=f32(1e-8))
        ref = lambda lr, t: CP.step_f32(orc, rule=rule, lr=lr, beta=f32(0.9), eps=f32(1e-8))
        keys = (("m", "s"),)
    return opt, dev_t, orc, run, ref, keys


@pytest.mark.parametrize("rule", ["ademamix", "lion", "momentum", "rmsprop", "adagrad", "mini"])
@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
def test_special_grads_reach_every_rule(rule, mode):
    """NaN, +-inf, +-0, subnormal and overflowing-square grads, no skip, two steps,
    through each rule's update: states equal up to NaN payloads, params likewise in
    fp32 mode and bit for bit as the stored bf16 + remainder pair."""
    rng = np.random.default_rng(zlib.crc32(f"rules/{rule}/{mode}".encode()))
    opt, dev_t, orc, run, ref, keys = _rule_setup(rule, mode, rng)
    lr_v = f32(1e-3)
    lr, step = scalar_f32(lr_v), scalar_i32(0)
    for t in (1, 2):
        for d, o, n in zip(dev_t, orc, RULE_SIZES):
            x, wide = grads_of(_grads(n, rng, False), torch.float32)
            d["g"].copy_(x)
            o.g = wide
        run(lr, step)
        with np.errstate(invalid="ignore", over="ignore", divide="ignore"):   # NaN / inf by design
            ref(lr_v, t)
    torch.cuda.synchronize()
    assert_guards_intact()
    for i, (d, o) in enumerate(zip(dev_t, orc)):
        for dk, ok in keys:
            assert _same_or_both_nan(host(d[dk]), getattr(o, ok)), (i, dk)
        if mode == "fp32":
            assert _same_or_both_nan(host(d["p"]), o.p), (i, "p")
        else:
            ohi, orem = OR.split(o.p)
            hi = host(d["p"].view(torch.int16)).view(np.uint16)
            assert np.array_equal(hi, ohi), (i, "bf16 half")
            assert np.array_equal(host(d["r"]), orem), (i, "remainder")
            assert np.all(np.isnan(OR.bf16_bits_to_f32(hi)[np.isnan(o.p)])), (i, "NaN -> bf16")
    assert int(step.item()) == 2 and opt.status() == 0
    opt.close()
