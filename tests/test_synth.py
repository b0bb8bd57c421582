"""The seeded synthetic workloads have the shapes, counts and value rules the
benchmark configurations state (CPU only).

GPT-2 small: 148 tensors, 124,439,808 elements, weight decay 0 on the layer
norms and biases (121,344 elements).  Llama-3-8B: 291 tensors, 8,030,261,248
elements.  The cosine schedule runs 1e-3 -> 1e-4 over 100 steps, the AMP
injection puts one non-finite grad in every 20-step window (+inf, -inf, NaN in
turn), the bf16 params with remainders never encode a NaN master, and the
Adam-mini block lengths satisfy the library's rule (1, numel, or a multiple of
8 dividing numel).
"""

import math

import numpy as np
import torch

import synth
from oracle import remainder as OR


def test_gpt2_small_list():
    specs = synth.gpt2_small()
    assert len(specs) == 148
    assert synth.total_numel(specs) == 124_439_808
    assert sum(s.numel for s in specs if s.wd == 0.0) == 121_344
    assert specs[0].shape == (50257, 768) and specs[1].shape == (1024, 768)
    assert all(s.wd == 0.0 for s in specs if s.name.endswith("bias") or "ln_" in s.name)


def test_llama3_8b_list():
    specs = synth.llama3_8b()
    assert len(specs) == 291
    assert synth.total_numel(specs) == 8_030_261_248
    names = [s.name for s in specs]
    assert names[0] == "tok_embeddings" and names[-1] == "output"
    assert all(s.wd == 0.1 for s in specs)


def test_cosine_schedule():
    lr = [synth.cosine_lr(s) for s in range(100)]
    assert math.isclose(lr[0], 1e-3, rel_tol=0, abs_tol=1e-18)
    assert math.isclose(lr[99], 1e-4, rel_tol=0, abs_tol=1e-18)
    assert all(a > b for a, b in zip(lr, lr[1:]))
    assert math.isclose(lr[0] + lr[99], lr[33] + lr[66], rel_tol=1e-12)  # symmetric about its middle


def test_amp_injection_one_per_window():
    inj = synth.amp_injection(100, 1 << 20, seed=3)
    assert len(inj) == 5
    windows = sorted(s // 20 for s in inj)
    assert windows == [0, 1, 2, 3, 4]
    vals = [inj[s][1] for s in sorted(inj)]
    assert vals[0] == math.inf and vals[1] == -math.inf and math.isnan(vals[2])
    assert vals[3] == math.inf and vals[4] == -math.inf
    assert all(0 <= i < (1 << 20) for i, _ in inj.values())


def test_bf16_params_with_remainders_have_finite_masters():
    hi, rem = synth.bf16_params_with_remainders(200_003, 0.02, seed=5, n_zeros=64)
    h = hi.view(torch.int16).numpy().view(np.uint16)
    r = rem.numpy()
    master = OR.join(h, r)
    assert np.all(np.isfinite(master))
    assert np.all(h[:64:2] == 0) and np.all(h[1:64:2] == 0x8000) and np.all(r[:64] == 0)
    zero = (h == 0) | (h == 0x8000)
    assert np.all(r[zero] >= 0)                      # a negative remainder under +-0 would be a NaN master
    assert np.any(r < 0)                             # elsewhere the remainder spans int16


def test_adam_mini_blocks_follow_the_library_rule():
    specs = synth.llama3_8b()
    blocks = synth.adam_mini_blocks(specs, dim=4096, n_heads=32)
    for s, b in zip(specs, blocks):
        assert s.numel % b == 0
        assert b in (1, s.numel) or b % 8 == 0
        if s.name in ("tok_embeddings", "output"):
            assert b == 1
        elif s.name.endswith(("attention.wq", "attention.wk")):
            assert b == 4096 * 4096 // 32
        else:
            assert b == s.numel


def test_seeds_and_draws_are_reproducible():
    seeds = {synth.grad_seed(7, s, k) for s in range(100) for k in range(148)}
    assert len(seeds) == 100 * 148
    a = synth.normal(4096, 1e-3, seed=11)
    b = synth.normal(4096, 1e-3, seed=11)
    assert torch.equal(a, b)
    assert not torch.equal(a, synth.normal(4096, 1e-3, seed=12))
    assert abs(float(a.std()) - 1e-3) < 1e-4
