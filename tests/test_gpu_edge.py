"""Degenerate plans for every entry point: an empty tensor list and a list of
zero-size tensors.  Nothing is read or written, but the step counter still
advances (a step that ran), exactly as for a plan with elements."""

import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu


def _zero(dtype=torch.float32):
    return torch.zeros(0, dtype=dtype, device="cuda")


def _plans(n):
    z = [_zero() for _ in range(n)]
    u8 = [_zero(torch.uint8) for _ in range(n)]
    return {
        "adamw": (FusedAdamW(z, z, z, z, [0.1] * n), lambda o, lr, st: o.step(lr, st)),
        "bf16_rem": (FusedAdamW([_zero(torch.bfloat16) for _ in range(n)], z, z, z, [0.1] * n,
                                mode="bf16_rem", param_rems=[_zero(torch.int16) for _ in range(n)]),
                     lambda o, lr, st: o.step(lr, st)),
        "ademamix": (FusedAdamW(z, z, z, z, [0.1] * n, exp_avg_slows=z),
                     lambda o, lr, st: o.step_ademamix(lr, st)),
        "lion": (FusedAdamW(z, z, z, None, [0.1] * n), lambda o, lr, st: o.step_lion(lr, st)),
        "adagrad": (FusedAdamW(z, z, z, None, [0.1] * n),
                    lambda o, lr, st: o.step_coupled("adagrad", lr, st)),
        "mini": (FusedAdamW(z, z, z, z, [0.1] * n, v_blocks=[1] * n),
                 lambda o, lr, st: o.step_mini(lr, st)),
        "q8": (FusedAdamW(z, z, u8, u8, [0.1] * n, mode="q8", absmax_m=z, absmax_v=z),
               lambda o, lr, st: o.step(lr, st)),
        "q4": (FusedAdamW(z, z, u8, u8, [0.1] * n, mode="q4", absmax_m=z, absmax_v=z),
               lambda o, lr, st: o.step(lr, st)),
        "amp": (FusedAdamW(z, z, z, z, [0.1] * n),
                lambda o, lr, st: o.step_amp(lr, st, zeros(1))),
    }


@pytest.mark.parametrize("n", [0, 3])
def test_degenerate_plans_count_steps(n):
    lr = torch.tensor([1e-3], device="cuda")
    for name, (opt, run) in _plans(n).items():
        st = zeros(1, torch.int32)
        for _ in range(3):
            run(opt, lr, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 3, name
        assert opt.status() == 0, name
        opt.close()


def test_plan_info_reports_the_launch_shape():
    """Every plan reports the CTA size of the kernel its step launches: the
    bulk-staged kernel (16 consumer warps + 1 producer warp), the 8-bit
    kernel (one 1024-thread CTA per SM with lane-private code tables) and the
    4-bit kernel (256 threads); the grid never exceeds the SM count times the
    CTAs that fit on one SM."""
    n = 1 << 22
    f = lambda dt=torch.float32: zeros(n, dt)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks = n // 256
    absq8 = zeros(blocks)
    absq4 = zeros(2 * blocks)
    cases = {
        "fp32": (FusedAdamW([f()], [f()], [f()], [f()], [0.1]), 544, 1),
        "q8": (FusedAdamW([f()], [f(torch.bfloat16)], [f(torch.uint8)], [f(torch.uint8)], [0.1],
                          mode="q8", absmax_m=[absq8], absmax_v=[absq8.clone()]), 1024, 1),
        "q4": (FusedAdamW([f()], [f(torch.bfloat16)], [zeros(n // 2, torch.uint8)],
                          [zeros(n // 2, torch.uint8)], [0.1], mode="q4",
                          absmax_m=[absq4], absmax_v=[absq4.clone()]), 256, 4),
    }
    for name, (opt, threads, per_sm) in cases.items():
        info = opt.info()
        assert info["block_threads"] == threads, name
        assert info["total_numel"] == n, name
        assert 1 <= info["grid_blocks"] <= per_sm * sms, name
        opt.close()


@pytest.mark.parametrize("start", [2**31 - 1, -7])
def test_step_counter_at_its_limits(start):
    """A step counter the caller left at INT32_MAX (t wraps) or set negative: the
    step ends (the bias corrections' power loop reads t as an unsigned 32-bit
    count, at most 32 rounds), the counter advances with 32-bit wrap-around, and
    the update is the oracle's at that unsigned t, where b^t = 0 and both bias
    corrections are 1 -- on the small kernel, the bulk kernel and the 8-bit one."""
    import numpy as np
    from oracle import adamw as OA
    from oracle import q8 as OQ
    f32 = OA.f32
    t_dev = (start + 1 + 2**31) % 2**32 - 2**31      # the counter after the step
    t_exp = (start + 1) % 2**32                      # the exponent the kernels use
    rng = np.random.default_rng(81)
    lr_v = f32(1e-3)
    hp = dict(beta1=f32(0.9), beta2=f32(0.999), eps=f32(1e-8))
    for sizes in ([5000], [4096 + 37 * i for i in range(20)]):   # small kernel, bulk kernel
        ps = [rng.normal(0, 0.02, n).astype(np.float32) for n in sizes]
        gs = [rng.normal(0, 1e-3, n).astype(np.float32) for n in sizes]
        d = [dict(p=dev(p), g=dev(g), m=zeros(p.size), v=zeros(p.size)) for p, g in zip(ps, gs)]
        opt = FusedAdamW([x["p"] for x in d], [x["g"] for x in d], [x["m"] for x in d],
                         [x["v"] for x in d], [f32(0.1)] * len(sizes))
        step = scalar_i32(start)
        opt.step(scalar_f32(lr_v), step, betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"])
        orc = [OA.Tensor(p=p.copy(), g=g, m=np.zeros(p.size, np.float32),
                         v=np.zeros(p.size, np.float32), wd=f32(0.1)) for p, g in zip(ps, gs)]
        OA.step_f32(orc, lr=lr_v, t=t_exp, **hp)
        torch.cuda.synchronize()
        assert int(step.item()) == t_dev and opt.status() == 0
        for x, o in zip(d, orc):
            assert bits_equal(host(x["p"]), o.p) and bits_equal(host(x["m"]), o.m)
            assert bits_equal(host(x["v"]), o.v)
        opt.close()
    # the 8-bit kernel's own launch
    n = 3000
    p, g = rng.normal(0, 0.02, n).astype(np.float32), rng.normal(0, 1e-3, n).astype(np.float32)
    nb = OQ.n_blocks(n)
    cm, cv = rng.integers(0, 256, n).astype(np.uint8), rng.integers(0, 256, n).astype(np.uint8)
    am, av = rng.uniform(0, 1e-3, nb).astype(np.float32), rng.uniform(0, 1e-6, nb).astype(np.float32)
    x = dict(p=dev(p), g=dev(g), cm=dev(cm), cv=dev(cv), am=dev(am), av=dev(av))
    opt = FusedAdamW([x["p"]], [x["g"]], [x["cm"]], [x["cv"]], [f32(0.01)], mode="q8",
                     absmax_m=[x["am"]], absmax_v=[x["av"]])
    step = scalar_i32(start)
    opt.step(scalar_f32(lr_v), step, betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"])
    OQ.step_f32(p, g, cm, cv, am, av, lr=lr_v, wd=f32(0.01), t=t_exp, **hp)
    torch.cuda.synchronize()
    assert int(step.item()) == t_dev and opt.status() == 0
    assert bits_equal(host(x["p"]), p) and np.array_equal(host(x["cm"]), cm)
    assert np.array_equal(host(x["cv"]), cv) and bits_equal(host(x["am"]), am)
    opt.close()
