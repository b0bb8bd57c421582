"""A small training loop through the library, against torch.optim.AdamW.

"FusedAdam & PyTorch Lightning AMP" compared a fused and an unfused AdamW on a
10x10 ``nn.Linear`` trained for a few epochs under AMP loss scaling.  Here the
same kind of loop runs twice from one seed: once with ``torch.optim.AdamW``
(float32, ``foreach=False``) behind the loss-scaling recipe GradScaler applies
-- scaled backward, skip on a non-finite grad, unscale, step -- with a fixed
scale, once with this library's AMP step (the loss scale and the
found-inf flag passed to the fused step, which unscales and skips by itself).
One batch carries an inf so both skip the same step.  The trajectories agree
to float32 rounding: torch's arithmetic differs from the strict-fp32 sequence
only in operation order.
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW

pytestmark = pytest.mark.gpu


def _model(seed):
    torch.manual_seed(seed)
    return torch.nn.Sequential(torch.nn.Linear(10, 10), torch.nn.Tanh(), torch.nn.Linear(10, 1)).cuda()


def _batches(n_batches, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    xs = [torch.randn(64, 10, generator=g, device="cuda") for _ in range(n_batches)]
    w = torch.randn(10, 1, generator=g, device="cuda")
    return [(x, torch.sin(x @ w)) for x in xs]


def test_training_loop_tracks_torch_adamw_under_amp():
    data = _batches(6 * 8, 17)                  # 6 epochs of 8 batches
    bad = 13                                    # this batch's loss gets an inf
    scale = 1024.0
    lr, wd = 1e-2, 0.1

    ref = _model(3)
    ropt = torch.optim.AdamW(ref.parameters(), lr=lr, weight_decay=wd, foreach=False)
    skipped_ref = 0

    ours = _model(3)
    params = list(ours.parameters())
    grads = [torch.zeros_like(p) for p in params]
    for p, g in zip(params, grads):
        p.grad = g                               # autograd accumulates into these buffers
    opt = FusedAdamW(params, grads, [torch.zeros_like(p) for p in params],
                     [torch.zeros_like(p) for p in params], [wd] * len(params))
    lr_d = torch.tensor([lr], device="cuda")
    step = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale_d = torch.tensor([scale], device="cuda")
    found = torch.zeros(1, device="cuda")

    losses_ref, losses_ours = [], []
    for i, (x, y) in enumerate(data):
        # torch.optim.AdamW behind fixed-scale loss scaling
        ropt.zero_grad(set_to_none=True)
        loss = torch.nn.functional.mse_loss(ref(x), y)
        if i == bad:
            loss = loss * float("inf")
        (loss * scale).backward()
        if all(torch.isfinite(p.grad).all() for p in ref.parameters()):
            for p in ref.parameters():
                p.grad.div_(scale)
            ropt.step()
        else:
            skipped_ref += 1
        losses_ref.append(float(loss.detach()))

        # the library: scaled backward, non-finite check, fused unscale + step
        for g in grads:
            g.zero_()
        loss2 = torch.nn.functional.mse_loss(ours(x), y)
        if i == bad:
            loss2 = loss2 * float("inf")
        (loss2 * scale).backward()
        assert all(p.grad.data_ptr() == g.data_ptr() for p, g in zip(params, grads))
        opt.check_nonfinite(found)
        opt.step(lr_d, step, grad_scale=scale_d, found_inf=found)
        losses_ours.append(float(loss2.detach()))

    torch.cuda.synchronize()
    assert int(step.item()) == len(data) - 1          # the inf batch was skipped
    assert skipped_ref == 1                           # by both
    fin = [k for k in range(len(data)) if k != bad]
    a, b = np.array(losses_ref)[fin], np.array(losses_ours)[fin]
    assert np.allclose(a, b, rtol=1e-4, atol=1e-7)
    assert b[-8:].mean() < 0.5 * b[:8].mean()         # it learns
    for p, q in zip(ref.parameters(), params):
        assert torch.allclose(p, q, rtol=1e-4, atol=1e-6)
