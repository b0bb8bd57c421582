"""adamw_step_amp: the non-finite check and the step in one cooperative launch.

Same AMP workload as the two-launch test (fp16 grads N(0,1e-3)*65536, loss scale
65536, one non-finite grad per 20-step window, 100 steps): bit-exact against the
strict-fp32 oracle, skipped steps leave everything untouched, the found-inf
output reports every skip, and results equal adamw_check_nonfinite +
adamw_step on the same plan type -- on all three routes adamw_step_amp takes
(the small kernel's fused variant, the cooperative fused kernel of mid-size or
misaligned plans, and the two launches past 6 Mi elements).
"""

import math

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW
from oracle import adamw as OA

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu
f32 = OA.f32
B1, B2, EPS = f32(0.9), f32(0.999), f32(1e-8)


def test_fused_amp_matches_oracle_and_skips():
    import synth
    n = 1 << 20
    rng = np.random.default_rng(31)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    p = dev(p0)
    g = zeros(n, torch.float16)
    m, v = zeros(n), zeros(n)
    opt = FusedAdamW([p], [g], [m], [v], [f32(0.1)])
    ref = OA.Tensor(p=p0.copy(), g=None, m=np.zeros(n, np.float32), v=np.zeros(n, np.float32),
                    wd=f32(0.1))
    inject = synth.amp_injection(100, n, seed=31)
    lr, step = torch.tensor([f32(0.1)], device="cuda"), zeros(1, torch.int32)
    scale, found = torch.tensor([65536.0], device="cuda"), torch.full((1,), 7.0, device="cuda")
    t = 0
    for s in range(100):
        x = (rng.normal(0, 1e-3, n) * 65536).astype(np.float16)
        if s in inject:
            i, val = inject[s]
            x[i] = val
        g.copy_(torch.from_numpy(x))
        ref.g = x.astype(np.float32)
        opt.step_amp(lr, step, found, betas=(B1, B2), eps=EPS, grad_scale=scale)
        ran = OA.step_f32([ref], lr=f32(0.1), beta1=B1, beta2=B2, eps=EPS, t=t + 1, grad_scale=65536.0)
        t += int(ran)
        torch.cuda.synchronize()
        assert found.item() == (0.0 if ran else 1.0), s
        assert int(step.item()) == t
        if s % 10 == 0 or s in inject or s == 99:
            assert np.array_equal(p.cpu().numpy().view(np.uint32), ref.p.view(np.uint32)), s
            assert np.array_equal(m.cpu().numpy().view(np.uint32), ref.m.view(np.uint32)), s
            assert np.array_equal(v.cpu().numpy().view(np.uint32), ref.v.view(np.uint32)), s
    assert t == 95 and opt.status() == 0


# the plan sizes adamw_step_amp routes three ways: the small kernel's fused
# variant (70,000 elements), the cooperative fused kernel of mid-size plans
# (3,000,000; and a small plan with a tensor off the 16-byte grid), and the
# two launches past 6 Mi elements (7,000,000)
CASES = {"small": (70_000, False), "mid": (3_000_000, False), "misaligned": (70_000, True),
         "big": (7_000_000, False)}


@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float16, torch.float32],
                         ids=["bf16", "f16", "f32"])
@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
@pytest.mark.parametrize("case", list(CASES))
def test_fused_amp_equals_two_launch_path(mode, case, gdtype):
    size, misalign = CASES[case]
    sizes = [1, 4099, size, 0, 257]
    rng = np.random.default_rng(32)
    sides = []
    for _ in range(2):
        rng_side = np.random.default_rng(33)
        st = []
        for i, n in enumerate(sizes):
            if mode == "fp32":
                pp = dev(rng_side.normal(0, 0.02, n).astype(np.float32))
                rr = None
            else:
                pp = to_dev(torch.from_numpy(rng_side.normal(0, 0.02, n).astype(np.float32)).to(torch.bfloat16))
                rr = dev(rng_side.integers(0, 1 << 15, n).astype(np.int16))
            # misaligned: tensor 1's m starts one float off the 16-byte grid
            mm = dev(np.zeros(n, np.float32), shift=1) if (misalign and i == 1) else zeros(n)
            st.append(dict(p=pp, r=rr, g=zeros(n, gdtype),
                           m=mm, v=zeros(n)))
        opt = FusedAdamW([d["p"] for d in st], [d["g"] for d in st], [d["m"] for d in st],
                         [d["v"] for d in st], [0.1, 0.0, 0.1, 0.0, 0.1], mode=mode,
                         param_rems=[d["r"] for d in st] if mode == "bf16_rem" else None)
        sides.append((st, opt, zeros(1, torch.int32),
                      zeros(1)))
    lr, scale = torch.tensor([1e-3], device="cuda"), torch.tensor([256.0], device="cuda")
    for it in range(6):
        xs = [torch.from_numpy((rng.normal(0, 1e-3, n) * 256).astype(np.float32)).to(gdtype)
              for n in sizes]
        if it == 3:
            xs[2][5] = math.inf
        for st, _, _, _ in sides:
            for d, x in zip(st, xs):
                d["g"].copy_(x)
        (st_a, opt_a, step_a, found_a), (st_b, opt_b, step_b, found_b) = sides
        opt_a.check_nonfinite(found_a)
        opt_a.step(lr, step_a, grad_scale=scale, found_inf=found_a)
        opt_b.step_amp(lr, step_b, found_b, grad_scale=scale)
        torch.cuda.synchronize()
        assert found_a.item() == found_b.item() == (1.0 if it == 3 else 0.0)
        assert int(step_a.item()) == int(step_b.item())
        for da, db in zip(st_a, st_b):
            for k in ("p", "r", "m", "v"):
                if da[k] is not None:
                    a = da[k].view(torch.int16 if da[k].element_size() == 2 else torch.int32)
                    b = db[k].view(torch.int16 if db[k].element_size() == 2 else torch.int32)
                    assert torch.equal(a, b), (it, k)
