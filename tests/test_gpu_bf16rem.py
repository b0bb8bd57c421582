"""GPU parity: bf16 params + int16 remainders (split/join and the step).

The split, the join and every step are bit-exact against the oracle: the
fp32 master the pair stands for is rebuilt, updated in the strict-fp32
sequence and split again ("Support store_param_remainders feature from Apex in
TE Fused Adam #1408", Description).
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW, adamw_bf16rem_join, adamw_bf16rem_split
from oracle import adamw as OA
from oracle import remainder as OR

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu
f32 = OA.f32
B1, B2, EPS = f32(0.9), f32(0.999), f32(1e-8)


def _special_bits():
    tops = [0x0000, 0x0001, 0x3F80, 0x7F7F, 0x7F80, 0x7FC0, 0x7FFF, 0x8000, 0x8001, 0xFF7F, 0xFF80, 0xFFFF]
    los = [0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF]
    return np.array([(t << 16) | lo for t in tops for lo in los], dtype=np.uint32)


@pytest.mark.parametrize("n", [1, 5, 4096, (1 << 22) + 3])
def test_split_join_bitexact(n):
    rng = np.random.default_rng(n)
    bits = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    sp = _special_bits()
    bits[: min(n, sp.size)] = sp[: min(n, sp.size)]
    master = dev(bits.view(np.float32))
    hi = empty(n, torch.int16)
    rem = empty(n, torch.int16)
    s = torch.cuda.current_stream().cuda_stream
    adamw_bf16rem_split(master.data_ptr(), hi.data_ptr(), rem.data_ptr(), n, s)
    back = empty(n, torch.float32)
    adamw_bf16rem_join(hi.data_ptr(), rem.data_ptr(), back.data_ptr(), n, s)
    torch.cuda.synchronize()
    ohi, orem = OR.split(bits)
    assert np.array_equal(host(hi).view(np.uint16), ohi)
    assert np.array_equal(host(rem), orem)
    # every master comes back bit for bit but a NaN, which comes back as the quiet NaN
    assert np.array_equal(host(back).view(np.uint32), OR.join(ohi, orem).view(np.uint32))
    nan = (bits & 0x7FFFFFFF) > 0x7F800000
    assert np.array_equal(host(back).view(np.uint32)[~nan], bits[~nan])
    assert np.all(host(back).view(np.uint32)[nan] == 0x7FC00000)


SIZES = [1, 7, 8, 9, 2049, 8192, 8193, 30001, 0, 64]


@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32, torch.float16])
def test_bf16rem_step_bitexact(gdtype):
    import synth
    rng = np.random.default_rng(7)
    his, rems, ms, vs, gs, oracle = [], [], [], [], [], []
    for i, n in enumerate(SIZES):
        hi_t, rem_t = synth.bf16_params_with_remainders(n, 0.02, seed=100 + i, device="cpu",
                                                        n_zeros=min(n, 64) if i == len(SIZES) - 1 else 0)
        hi_bits = hi_t.view(torch.int16).numpy().view(np.uint16).copy()
        rem_np = rem_t.numpy().copy()
        his.append(to_dev(hi_t))
        rems.append(to_dev(rem_t))
        m = rng.normal(0, 1e-4, n).astype(np.float32)
        v = (rng.normal(0, 1e-4, n) ** 2).astype(np.float32)
        ms.append(dev(m))
        vs.append(dev(v))
        gs.append(empty(n, gdtype))
        oracle.append(OA.Tensor(p=OR.join(hi_bits, rem_np), g=None, m=m.copy(), v=v.copy(),
                                wd=f32(0.1)))
    opt = FusedAdamW(his, gs, ms, vs, [f32(0.1)] * len(SIZES), mode="bf16_rem", param_rems=rems)
    lr, step = scalar_f32(f32(3e-4)), scalar_i32(0)
    for t in range(1, 6):
        for g, o in zip(gs, oracle):
            tg, wide = grads_of(rng.normal(0, 1e-4, g.numel()).astype(np.float32), gdtype)
            g.copy_(tg)
            o.g = wide
        opt.step(lr, step, betas=(B1, B2), eps=EPS)
        OA.step_f32(oracle, lr=f32(3e-4), beta1=B1, beta2=B2, eps=EPS, t=t)
        torch.cuda.synchronize()
        for i, (h, r, m, v, o) in enumerate(zip(his, rems, ms, vs, oracle)):
            ohi, orem = OR.split(o.p)
            assert np.array_equal(host(h).view(np.uint16), ohi), f"tensor {i} bf16 step {t}"
            assert np.array_equal(host(r), orem), f"tensor {i} rem step {t}"
            assert bits_equal(host(m), o.m), f"tensor {i} m: {first_mismatch(host(m), o.m)}"
            assert bits_equal(host(v), o.v), f"tensor {i} v: {first_mismatch(host(v), o.v)}"
    assert int(step.item()) == 5


def test_bf16rem_bulk_path_with_twenty_tensors():
    """20 tensors (more than a small plan takes): the bulk-staged kernel, bit-exact."""
    import synth
    rng = np.random.default_rng(17)
    sizes = SIZES + [16385, 3, 40000, 1 << 15, 255, 8200, 1, 999, 4096, 12345]
    his, rems, ms, vs, gs, oracle = [], [], [], [], [], []
    for i, n in enumerate(sizes):
        hi_t, rem_t = synth.bf16_params_with_remainders(n, 0.02, seed=200 + i, device="cpu")
        hi_bits = hi_t.view(torch.int16).numpy().view(np.uint16).copy()
        rem_np = rem_t.numpy().copy()
        his.append(to_dev(hi_t))
        rems.append(to_dev(rem_t))
        m = rng.normal(0, 1e-4, n).astype(np.float32)
        v = (rng.normal(0, 1e-4, n) ** 2).astype(np.float32)
        ms.append(dev(m))
        vs.append(dev(v))
        gs.append(empty(n, torch.bfloat16))
        oracle.append(OA.Tensor(p=OR.join(hi_bits, rem_np), g=None, m=m.copy(), v=v.copy(),
                                wd=f32(0.1)))
    opt = FusedAdamW(his, gs, ms, vs, [f32(0.1)] * len(sizes), mode="bf16_rem", param_rems=rems)
    assert opt.info()["block_threads"] == 544
    lr, step = scalar_f32(f32(3e-4)), scalar_i32(0)
    for t in range(1, 4):
        for g, o in zip(gs, oracle):
            tg, wide = grads_of(rng.normal(0, 1e-4, g.numel()).astype(np.float32), torch.bfloat16)
            g.copy_(tg)
            o.g = wide
        opt.step(lr, step, betas=(B1, B2), eps=EPS)
        OA.step_f32(oracle, lr=f32(3e-4), beta1=B1, beta2=B2, eps=EPS, t=t)
        torch.cuda.synchronize()
        assert_guards_intact()
        for i, (h, r, m, v, o) in enumerate(zip(his, rems, ms, vs, oracle)):
            ohi, orem = OR.split(o.p)
            assert np.array_equal(host(h).view(np.uint16), ohi), f"tensor {i} bf16 step {t}"
            assert np.array_equal(host(r), orem), f"tensor {i} rem step {t}"
            assert bits_equal(host(m), o.m), f"tensor {i} m"
            assert bits_equal(host(v), o.v), f"tensor {i} v"
