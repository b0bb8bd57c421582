"""Degenerate plans for every entry point: an empty tensor list and a list of
zero-size tensors.  Nothing is read or written, but the step counter still
advances (a step that ran), exactly as for a plan with elements."""

import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW

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
                lambda o, lr, st: o.step_amp(lr, st, torch.zeros(1, device="cuda"))),
    }


@pytest.mark.parametrize("n", [0, 3])
def test_degenerate_plans_count_steps(n):
    lr = torch.tensor([1e-3], device="cuda")
    for name, (opt, run) in _plans(n).items():
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(3):
            run(opt, lr, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 3, name
        assert opt.status() == 0, name
        opt.close()
