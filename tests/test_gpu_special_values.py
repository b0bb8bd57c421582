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
