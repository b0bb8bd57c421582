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
