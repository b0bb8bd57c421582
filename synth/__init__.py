"""Seeded synthetic inputs for the AdamW step workloads.

Shared by the tests, ``bench.py`` and ``smoke()``; imported by neither the GPU
library nor the oracle's arithmetic.  This module holds shapes, seeds, value
distributions and the learning-rate schedule of the workloads -- none of the
optimizer's arithmetic.  Random values come from ``torch.Generator`` (seeded,
on the device the tensor lives on); a test that needs the same values on the
oracle copies the generated inputs to the host.

Workloads (sizes in elements):
  single      one fp32 tensor of 1,048,576; p~N(0,0.02), g~N(0,1e-3);
              lr = wd = 0.1, betas (0.9, 0.999), eps 1e-8; 10 steps.
  gpt2_small  148 fp32 tensors, 124,439,808 elements (GPT-2 small layout);
              wd 0 on layer-norm weights/biases and on all biases, else 0.1;
              lr from a device scalar on a cosine schedule 1e-3 -> 1e-4 over
              100 steps.
  amp         the single-tensor shapes with fp16 grads N(0,1e-3)*65536 and a
              fixed loss scale 65536; in every window of 20 steps one seeded
              step gets one non-finite element (+inf, -inf, NaN in turn);
              100 steps.
  q8          one flat fp32 tensor of 2**30, bf16 grads N(0,1e-3), 8-bit
              blockwise m, v from zero state; lr 1e-3, wd 0.01; 20 steps.
  llama3_8b   291 tensors, 8,030,261,248 elements (Llama-3-8B layout) as
              bf16 params + int16 remainders, bf16 grads N(0,1e-4), fp32 m, v;
              lr 3e-4, wd 0.1 on every tensor; 5 steps.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple[int, ...]
    wd: float

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


def gpt2_small(wd: float = 0.1) -> list[TensorSpec]:
    """GPT-2 small parameter list; layer norms and biases get wd = 0."""
    d, ff, vocab, ctx = 768, 3072, 50257, 1024
    out = [TensorSpec("wte", (vocab, d), wd), TensorSpec("wpe", (ctx, d), wd)]
    for i in range(12):
        h = f"h.{i}."
        out += [
            TensorSpec(h + "ln_1.weight", (d,), 0.0),
            TensorSpec(h + "ln_1.bias", (d,), 0.0),
            TensorSpec(h + "attn.c_attn.weight", (d, 3 * d), wd),
            TensorSpec(h + "attn.c_attn.bias", (3 * d,), 0.0),
            TensorSpec(h + "attn.c_proj.weight", (d, d), wd),
            TensorSpec(h + "attn.c_proj.bias", (d,), 0.0),
            TensorSpec(h + "ln_2.weight", (d,), 0.0),
            TensorSpec(h + "ln_2.bias", (d,), 0.0),
            TensorSpec(h + "mlp.c_fc.weight", (d, ff), wd),
            TensorSpec(h + "mlp.c_fc.bias", (ff,), 0.0),
            TensorSpec(h + "mlp.c_proj.weight", (ff, d), wd),
            TensorSpec(h + "mlp.c_proj.bias", (d,), 0.0),
        ]
    out += [TensorSpec("ln_f.weight", (d,), 0.0), TensorSpec("ln_f.bias", (d,), 0.0)]
    return out


def llama3_8b(wd: float = 0.1) -> list[TensorSpec]:
    """Llama-3-8B parameter list; every tensor gets the same wd."""
    d, kv, ff, vocab = 4096, 1024, 14336, 128256
    out = [TensorSpec("tok_embeddings", (vocab, d), wd)]
    for i in range(32):
        h = f"layers.{i}."
        out += [
            TensorSpec(h + "attention.wq", (d, d), wd),
            TensorSpec(h + "attention.wk", (kv, d), wd),
            TensorSpec(h + "attention.wv", (kv, d), wd),
            TensorSpec(h + "attention.wo", (d, d), wd),
            TensorSpec(h + "feed_forward.w1", (ff, d), wd),
            TensorSpec(h + "feed_forward.w3", (ff, d), wd),
            TensorSpec(h + "feed_forward.w2", (d, ff), wd),
            TensorSpec(h + "attention_norm", (d,), wd),
            TensorSpec(h + "ffn_norm", (d,), wd),
        ]
    out += [TensorSpec("norm", (d,), wd), TensorSpec("output", (vocab, d), wd)]
    return out


def adam_mini_blocks(specs: list[TensorSpec], dim: int, n_heads: int) -> list[int]:
    """Adam-mini block length per tensor by parameter name, as the AdamWMini
    listing of "Adam-mini <> DTensor" partitions a model: embeddings and the
    output layer keep one v per element, query and key weights one per head
    (dim*dim/n_heads elements), every other tensor one v for the whole tensor."""
    out = []
    for s in specs:
        if any(k in s.name for k in ("embed", "embd", "wte", "lm_head", "output")):
            out.append(1)
        elif any(k in s.name for k in ("wq", "wk", "q_proj", "k_proj")):
            out.append(dim * dim // n_heads)
        else:
            out.append(s.numel)
    return out


def total_numel(specs: list[TensorSpec]) -> int:
    return sum(s.numel for s in specs)


def cosine_lr(s: int, total: int = 100, lr_max: float = 1e-3, lr_min: float = 1e-4) -> float:
    """Cosine schedule value at step s (0-based): lr_max at s=0, lr_min at s=total-1.

    The pages ask for a tensor learning rate so that a per-step schedule costs
    nothing ("4 bit Adam should support non constant lr"); they give no
    formula, so the plain half-cosine is used, in float64.
    """
    return lr_min + 0.5 * (lr_max - lr_min) * (1.0 + math.cos(math.pi * s / (total - 1)))


def gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(n: int, std: float, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """n samples of N(0, std**2), drawn in float32 then cast to dtype."""
    x = torch.randn(n, generator=gen(seed, device), device=device, dtype=torch.float32)
    x.mul_(std)
    return x if dtype == torch.float32 else x.to(dtype)


def grad_seed(base: int, step: int, tensor: int = 0) -> int:
    """Seed of the grads of one tensor at one (0-based) step."""
    return (base * 1_000_003 + step * 7919 + tensor * 104_729) & 0x7FFFFFFF


def bf16_params_with_remainders(n: int, std: float, seed: int, device="cpu",
                                n_zeros: int = 0) -> tuple[torch.Tensor, torch.Tensor]:
    """A bf16 model param and an int16 remainder array, drawn directly.

    The bf16 half is N(0, std**2) rounded by torch; the remainder is uniform
    over int16, except where the bf16 half is +0 or -0, where it is drawn in
    [0, 32767] (a negative remainder under a zero would stand for a NaN
    master).  The first ``n_zeros`` elements are forced to +0 / -0 in turn
    with remainder 0, so that exact zeros are exercised.
    """
    g = gen(seed, device)
    hi = (torch.randn(n, generator=g, device=device) * std).to(torch.bfloat16)
    rem = torch.randint(-32768, 32768, (n,), generator=g, device=device, dtype=torch.int32)
    hi_bits = hi.view(torch.int16)
    if n_zeros:
        k = min(n_zeros, n)
        z = torch.zeros(k, dtype=torch.int16, device=device)
        z[1::2] = -32768  # 0x8000 = -0.0
        hi_bits[:k] = z
        rem[:k] = 0
    is_zero = (hi_bits == 0) | (hi_bits == -32768)
    rem = torch.where(is_zero, rem & 0x7FFF, rem).to(torch.int16)
    return hi, rem


def amp_injection(n_steps: int, numel: int, seed: int, window: int = 20) -> dict[int, tuple[int, float]]:
    """{step: (element index, value)} -- one non-finite grad per window of steps.

    Values cycle +inf, -inf, NaN over successive windows.
    """
    g = gen(seed, "cpu")
    vals = [math.inf, -math.inf, math.nan]
    out = {}
    for w in range(n_steps // window):
        s = w * window + int(torch.randint(0, window, (1,), generator=g))
        i = int(torch.randint(0, numel, (1,), generator=g))
        out[s] = (i, vals[w % 3])
    return out
