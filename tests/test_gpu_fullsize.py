"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times.

The workloads are built by bench.py's own classes (same plans, same layout,
same grids).  Each step gets new seeded device grads; a fixed sample of
elements -- the first and last elements of every tensor plus random windows
(whole 256-element blocks on the 8-bit path) -- is followed through every step
by the strict-fp32 oracle, from inputs copied off the device before the library
touches them.  Sampled outputs must match bit for bit, and the fp32 params must
stay within the float64 definition's tolerance.
"""

import gc

import numpy as np
import pytest
import torch

import bench
import synth
from oracle import adamw as OA
from oracle import q8 as OQ
from oracle import remainder as OR

pytestmark = pytest.mark.gpu


def _free_gib():
    free, _ = torch.cuda.mem_get_info()
    return free / 2 ** 30


def _windows(numels, rng, edge=64, n_rand=24, width=256, align=1):
    """Per tensor: sorted element indices (edges + random windows)."""
    out = []
    for n in numels:
        idx = set(range(min(edge, n))) | set(range(max(0, n - edge), n))
        for _ in range(n_rand if n > 4 * width else 0):
            s = int(rng.integers(0, n - width)) // align * align
            idx |= set(range(s, s + width))
        out.append(np.array(sorted(idx), dtype=np.int64))
    return out


def _take(t, idx):
    return t.view(-1)[torch.from_numpy(idx).to(t.device)]


def _cleanup():
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_gpt2_small_full_size_cosine_lr_sampled():
    """148 tensors, 124,439,808 elements, lr from the device cosine table, 100 steps."""
    w = bench.Gpt2Small()
    try:
        rng = np.random.default_rng(21)
        idx = _windows([p.numel() for p in w.ps], rng)
        orc = [OA.Tensor(p=_take(p, i).cpu().numpy(), g=None, m=_take(m, i).cpu().numpy(),
                         v=_take(v, i).cpu().numpy(), wd=s.wd)
               for p, m, v, i, s in zip(w.ps, w.ms, w.vs, idx, w.specs)]
        ref = [OA.Tensor(p=o.p.astype(np.float64), g=None, m=o.m.astype(np.float64),
                         v=o.v.astype(np.float64), wd=o.wd) for o in orc]
        for s in range(100):
            gs = w.step_grads(s)
            for k, g in enumerate(gs):
                g.copy_(synth.normal(g.numel(), 1e-3, synth.grad_seed(7, s, k), "cuda"))
            for o, r, g, i in zip(orc, ref, gs, idx):
                o.g = _take(g, i).cpu().numpy()
                r.g = o.g.astype(np.float64)
            w.step(s)
            lr = float(w.lr_table[s % 100].item())
            OA.step_f32(orc, lr=lr, beta1=OA.f32(0.9), beta2=OA.f32(0.999), eps=OA.f32(1e-8), t=s + 1)
            OA.step_fp64(ref, lr=lr, beta1=OA.f32(0.9), beta2=OA.f32(0.999), eps=OA.f32(1e-8), t=s + 1)
            if s in (0, 1, 50, 99):
                torch.cuda.synchronize()
                for k, (p, m, v, i, o) in enumerate(zip(w.ps, w.ms, w.vs, idx, orc)):
                    assert np.array_equal(_take(p, i).cpu().numpy().view(np.uint32), o.p.view(np.uint32)), (s, k)
                    assert np.array_equal(_take(m, i).cpu().numpy().view(np.uint32), o.m.view(np.uint32)), (s, k)
                    assert np.array_equal(_take(v, i).cpu().numpy().view(np.uint32), o.v.view(np.uint32)), (s, k)
        assert int(w.step_dev.item()) == 100
        assert w.status() == 0
        worst = max(np.max(np.abs(o.p.astype(np.float64) - r.p)) for o, r in zip(orc, ref))
        assert worst <= 5e-5
    finally:
        del w
        _cleanup()


def _division_rule_gap(kernel_codes, x, absmax, block, table, thr):
    """The kernel's codes (normalised as x * fl(1/A)) against the plain division
    rule, the nearest code of fl(x / A), on the same pre-quantisation state x of
    the sampled blocks: every code that differs is off by one and the exact
    ratio x / A lies within 2.5 ulp of the threshold between the two codes.
    Returns the number of differing codes."""
    from oracle import qmap as QM
    x = np.asarray(x, np.float32)
    a = np.repeat(np.asarray(absmax, np.float32), block)[: x.size]
    nz = a > 0
    div = np.asarray(kernel_codes).astype(np.int64).copy()
    div[nz] = QM.quantize((x[nz] / a[nz]).astype(np.float32), table, thr)
    k = np.asarray(kernel_codes).astype(np.int64)
    bad = np.nonzero(k != div)[0]
    if bad.size:
        assert np.all(np.abs(k[bad] - div[bad]) == 1)
        t = thr[np.minimum(k[bad], div[bad])].astype(np.float64)
        ulp = np.nextafter(np.abs(t).astype(np.float32), np.float32(np.inf)).astype(np.float64) - np.abs(t)
        exact = x[bad].astype(np.float64) / a[bad].astype(np.float64)
        assert np.all(np.abs(exact - t) <= 2.5 * ulp)
    return int(bad.size)


def test_q8_full_size_2e30_sampled_blocks():
    """One 2^30 fp32 tensor, 8-bit m and v, bf16 grads, lr 1e-3, wd 0.01, 20 steps."""
    if _free_gib() < 12:
        pytest.skip("needs ~9 GiB of free device memory")
    w = bench.Q8()
    try:
        rng = np.random.default_rng(22)
        n = w.n_params
        blocks = np.unique(np.concatenate([[0, 1, n // 256 - 1],
                                           rng.integers(0, n // 256, 64)]))
        idx = (blocks[:, None] * 256 + np.arange(256)[None, :]).ravel()
        bidx = torch.from_numpy(blocks).cuda()
        p = _take(w.p, idx).cpu().numpy()
        cm = _take(w.cm, idx).cpu().numpy()
        cv = _take(w.cv, idx).cpu().numpy()
        am = w.am[bidx].cpu().numpy()
        av = w.av[bidx].cpu().numpy()
        maps = OQ.Maps()
        gap = 0
        for s in range(20):
            w.g.copy_(synth.normal(n, 1e-3, synth.grad_seed(8, s), "cuda", torch.bfloat16))
            g = _take(w.g, idx).float().cpu().numpy()
            w.step(s)
            sc = OA.f32_scalars(lr=OA.f32(1e-3), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                                eps=OA.f32(1e-8), t=s + 1)
            _, m1, v1 = OA.elementwise_f32(p, g, OQ.dequantize(cm, am, maps.smap),
                                           OQ.dequantize(cv, av, maps.umap), sc,
                                           OA.decay_f32(sc.lr, OA.f32(0.01)))
            OQ.step_f32(p, g, cm, cv, am, av, lr=OA.f32(1e-3), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                        eps=OA.f32(1e-8), wd=OA.f32(0.01), t=s + 1, maps=maps)
            torch.cuda.synchronize()
            gap += _division_rule_gap(_take(w.cm, idx).cpu().numpy(), m1, am, 256, maps.smap, maps.sthr)
            gap += _division_rule_gap(_take(w.cv, idx).cpu().numpy(), v1, av, 256, maps.umap, maps.uthr)
        print(f"8-bit codes that differ from the division rule: {gap} of {2 * 20 * idx.size}")
        assert gap <= 1e-4 * 2 * 20 * idx.size
        assert np.array_equal(_take(w.p, idx).cpu().numpy().view(np.uint32), p.view(np.uint32))
        assert np.array_equal(_take(w.cm, idx).cpu().numpy(), cm)
        assert np.array_equal(_take(w.cv, idx).cpu().numpy(), cv)
        assert np.array_equal(w.am[bidx].cpu().numpy().view(np.uint32), am.view(np.uint32))
        assert np.array_equal(w.av[bidx].cpu().numpy().view(np.uint32), av.view(np.uint32))
        assert int(w.step_dev.item()) == 20
    finally:
        del w
        _cleanup()


def test_llama3_8b_bf16_remainders_full_size_sampled():
    """291 tensors, 8,030,261,248 elements as bf16 + int16 remainders, 5 steps."""
    if _free_gib() < 120:
        pytest.skip("needs ~115 GiB of free device memory")
    w = bench.Llama3()
    try:
        hs, rs, gs, ms, vs = w._views
        rng = np.random.default_rng(23)
        idx = _windows([h.numel() for h in hs], rng, n_rand=4)
        orc = []
        for h, r, m, v, i, spec in zip(hs, rs, ms, vs, idx, w.specs):
            hi = _take(h.view(torch.int16), i).cpu().numpy().view(np.uint16)
            rem = _take(r, i).cpu().numpy()
            orc.append(OA.Tensor(p=OR.join(hi, rem), g=None, m=_take(m, i).cpu().numpy(),
                                 v=_take(v, i).cpu().numpy(), wd=spec.wd))
        for s in range(5):
            for k, g in enumerate(gs):
                g.copy_(synth.normal(g.numel(), 1e-4, synth.grad_seed(9, s, k), "cuda", torch.bfloat16))
            for o, g, i in zip(orc, gs, idx):
                o.g = _take(g, i).float().cpu().numpy()
            w.step(s)
            OA.step_f32(orc, lr=OA.f32(3e-4), beta1=OA.f32(0.9), beta2=OA.f32(0.999), eps=OA.f32(1e-8),
                        t=s + 1)
        torch.cuda.synchronize()
        for k, (h, r, m, v, i, o) in enumerate(zip(hs, rs, ms, vs, idx, orc)):
            ohi, orem = OR.split(o.p)
            assert np.array_equal(_take(h.view(torch.int16), i).cpu().numpy().view(np.uint16), ohi), k
            assert np.array_equal(_take(r, i).cpu().numpy(), orem), k
            assert np.array_equal(_take(m, i).cpu().numpy().view(np.uint32), o.m.view(np.uint32)), k
            assert np.array_equal(_take(v, i).cpu().numpy().view(np.uint32), o.v.view(np.uint32)), k
        assert int(w.step_dev.item()) == 5
        assert w.opt.status() == 0
    finally:
        del w
        _cleanup()


def test_single_tensor_beyond_2e31_elements():
    """One fp32 tensor of 2^31 + 4097 elements: 64-bit indexing inside a tensor and a
    ragged tail; sampled windows at both ends and across element 2^31."""
    n = (1 << 31) + 4097
    if _free_gib() < 40:
        pytest.skip("needs ~35 GiB of free device memory")
    from adamw_optimizer_step_tensor_gb300 import FusedAdamW
    try:
        p = synth.normal(n, 0.02, 61, "cuda")
        g = torch.empty(n, device="cuda")
        m = torch.zeros(n, device="cuda")
        v = torch.zeros(n, device="cuda")
        opt = FusedAdamW([p], [g], [m], [v], [OA.f32(0.1)])
        idx = np.concatenate([np.arange(0, 4096), np.arange((1 << 31) - 2048, (1 << 31) + 2048),
                              np.arange(n - 4096, n)]).astype(np.int64)
        orc = OA.Tensor(p=_take(p, idx).cpu().numpy(), g=None, m=np.zeros(idx.size, np.float32),
                        v=np.zeros(idx.size, np.float32), wd=OA.f32(0.1))
        lr, step = torch.tensor([OA.f32(1e-3)], device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
        for s in range(3):
            g.copy_(synth.normal(n, 1e-3, 62 + s, "cuda"))
            orc.g = _take(g, idx).cpu().numpy()
            opt.step(lr, step)
            OA.step_f32([orc], lr=OA.f32(1e-3), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                        eps=OA.f32(1e-8), t=s + 1)
        torch.cuda.synchronize()
        assert np.array_equal(_take(p, idx).cpu().numpy().view(np.uint32), orc.p.view(np.uint32))
        assert np.array_equal(_take(m, idx).cpu().numpy().view(np.uint32), orc.m.view(np.uint32))
        assert np.array_equal(_take(v, idx).cpu().numpy().view(np.uint32), orc.v.view(np.uint32))
        assert int(step.item()) == 3 and opt.status() == 0
    finally:
        _cleanup()


def test_bf16rem_tensor_beyond_2e31_elements():
    """One bf16 + int16-remainder tensor of 2^31 + 4097 elements (bf16 grads): windows
    at both ends and across element 2^31, bit-exact over 3 steps."""
    n = (1 << 31) + 4097
    if _free_gib() < 45:
        pytest.skip("needs ~40 GiB of free device memory")
    from adamw_optimizer_step_tensor_gb300 import FusedAdamW
    try:
        hi, rem = synth.bf16_params_with_remainders(n, 0.02, 69, "cuda", n_zeros=64)
        g = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        m = torch.zeros(n, device="cuda")
        v = torch.zeros(n, device="cuda")
        opt = FusedAdamW([hi], [g], [m], [v], [OA.f32(0.1)], mode="bf16_rem", param_rems=[rem])
        idx = np.concatenate([np.arange(0, 4096), np.arange((1 << 31) - 2048, (1 << 31) + 2048),
                              np.arange(n - 4096, n)]).astype(np.int64)
        orc = OA.Tensor(p=OR.join(_take(hi.view(torch.int16), idx).cpu().numpy().view(np.uint16),
                                  _take(rem, idx).cpu().numpy()),
                        g=None, m=np.zeros(idx.size, np.float32), v=np.zeros(idx.size, np.float32),
                        wd=OA.f32(0.1))
        lr, step = torch.tensor([OA.f32(3e-4)], device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
        for s in range(3):
            g.copy_(synth.normal(n, 1e-4, 70 + s, "cuda", torch.bfloat16))
            orc.g = _take(g, idx).float().cpu().numpy()
            opt.step(lr, step)
            OA.step_f32([orc], lr=OA.f32(3e-4), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                        eps=OA.f32(1e-8), t=s + 1)
        torch.cuda.synchronize()
        ohi, orem = OR.split(orc.p)
        assert np.array_equal(_take(hi.view(torch.int16), idx).cpu().numpy().view(np.uint16), ohi)
        assert np.array_equal(_take(rem, idx).cpu().numpy(), orem)
        assert np.array_equal(_take(m, idx).cpu().numpy().view(np.uint32), orc.m.view(np.uint32))
        assert np.array_equal(_take(v, idx).cpu().numpy().view(np.uint32), orc.v.view(np.uint32))
        assert int(step.item()) == 3 and opt.status() == 0
    finally:
        _cleanup()


def test_adam_mini_block_beyond_2e31_elements():
    """One Adam-mini block (v shared by the whole tensor) of 2^31 + 4097 elements,
    bf16 grads, 2 steps: the reduction over the block's 131,073 chunks and the update
    across element 2^31.  The oracle's block sum is taken piece by piece in float64
    on the host (its order is free); v must match to one ulp per step, m bit for bit,
    and the sampled params to the error one v ulp can cause."""
    from oracle import mini as M
    n = (1 << 31) + 4097
    if _free_gib() < 35:
        pytest.skip("needs ~30 GiB of free device memory")
    from adamw_optimizer_step_tensor_gb300 import FusedAdamW
    try:
        p = synth.normal(n, 0.02, 76, "cuda")
        g = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        m = torch.zeros(n, device="cuda")
        v = torch.zeros(1, device="cuda")
        opt = FusedAdamW([p], [g], [m], [v], [OA.f32(0.1)], v_blocks=[n])
        idx = np.concatenate([np.arange(0, 4096), np.arange((1 << 31) - 2048, (1 << 31) + 2048),
                              np.arange(n - 4096, n)]).astype(np.int64)
        orc = M.Tensor(p=_take(p, idx).cpu().numpy(), g=None, m=np.zeros(idx.size, np.float32),
                       v=np.zeros(1, np.float32), wd=OA.f32(0.1), block=idx.size)
        lr = OA.f32(3e-4)
        lr_dev, step = torch.tensor([lr], device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
        piece = 1 << 27
        for s in range(2):
            g.copy_(synth.normal(n, 1e-3, 77 + s, "cuda", torch.bfloat16))
            total = sum(M.block_sum_sq(g[a:a + piece].float().cpu().numpy()) for a in range(0, n, piece))
            orc.g = _take(g, idx).float().cpu().numpy()
            opt.step_mini(lr_dev, step, betas=(OA.f32(0.9), OA.f32(0.999)), eps=OA.f32(1e-8))
            M.step_f32([orc], lr=lr, beta1=OA.f32(0.9), beta2=OA.f32(0.999), eps=OA.f32(1e-8),
                       t=s + 1, means=[np.array([M.mean_from_sum(total, n)])])
        torch.cuda.synchronize()
        vd = v.cpu().numpy()
        assert abs(int(vd.view(np.int32)[0]) - int(orc.v.view(np.int32)[0])) <= 2, (vd, orc.v)
        assert np.array_equal(_take(m, idx).cpu().numpy().view(np.uint32), orc.m.view(np.uint32))
        pd = _take(p, idx).cpu().numpy().astype(np.float64)
        r_scale = np.abs(orc.m).astype(np.float64) / np.sqrt(float(orc.v[0]))
        tol = 2.0 ** -22 * (np.abs(orc.p) + lr * r_scale * 4) * 2
        assert np.all(np.abs(pd - orc.p) <= tol)
        assert int(step.item()) == 2 and opt.status() == 0
    finally:
        _cleanup()


def _blocks_beyond_2e31(n, block, rng):
    """Whole blocks sampled at both ends of an n-element tensor, across element
    2^31 and at random, sorted; the partial last block's index comes last."""
    full = n // block
    pivot = (1 << 31) // block
    blocks = np.unique(np.concatenate([np.arange(0, 4), np.arange(pivot - 4, pivot + 4),
                                       np.arange(full - 4, full), rng.integers(0, full, 16)]))
    idx = np.concatenate([(blocks[:, None] * block + np.arange(block)[None, :]).ravel(),
                          np.arange(full * block, n)]).astype(np.int64)
    return np.concatenate([blocks, [full]]).astype(np.int64), idx


def test_q8_tensor_beyond_2e31_elements():
    """One fp32 tensor of 2^31 + 4097 elements with 8-bit m and v (bf16 grads): whole
    blocks across element 2^31, at both ends and at random, plus the 1-element last
    block, bit-exact over 3 steps."""
    n = (1 << 31) + 4097
    if _free_gib() < 30:
        pytest.skip("needs ~25 GiB of free device memory")
    from adamw_optimizer_step_tensor_gb300 import FusedAdamW
    try:
        rng = np.random.default_rng(63)
        nb = (n + 255) // 256
        w_p = synth.normal(n, 0.02, 64, "cuda")
        w_g = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        cm = torch.zeros(n, dtype=torch.uint8, device="cuda")
        cv = torch.zeros(n, dtype=torch.uint8, device="cuda")
        am, av = torch.zeros(nb, device="cuda"), torch.zeros(nb, device="cuda")
        opt = FusedAdamW([w_p], [w_g], [cm], [cv], [OA.f32(0.01)], mode="q8",
                         absmax_m=[am], absmax_v=[av])
        bidx, idx = _blocks_beyond_2e31(n, 256, rng)
        tb = torch.from_numpy(bidx).cuda()
        p, ocm, ocv = _take(w_p, idx).cpu().numpy(), _take(cm, idx).cpu().numpy(), _take(cv, idx).cpu().numpy()
        oam, oav = am[tb].cpu().numpy(), av[tb].cpu().numpy()
        maps = OQ.Maps()
        lr, step = torch.tensor([OA.f32(1e-3)], device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
        for s in range(3):
            w_g.copy_(synth.normal(n, 1e-3, 65 + s, "cuda", torch.bfloat16))
            g = _take(w_g, idx).float().cpu().numpy()
            opt.step(lr, step)
            OQ.step_f32(p, g, ocm, ocv, oam, oav, lr=OA.f32(1e-3), beta1=OA.f32(0.9),
                        beta2=OA.f32(0.999), eps=OA.f32(1e-8), wd=OA.f32(0.01), t=s + 1, maps=maps)
        torch.cuda.synchronize()
        assert np.array_equal(_take(w_p, idx).cpu().numpy().view(np.uint32), p.view(np.uint32))
        assert np.array_equal(_take(cm, idx).cpu().numpy(), ocm)
        assert np.array_equal(_take(cv, idx).cpu().numpy(), ocv)
        assert np.array_equal(am[tb].cpu().numpy().view(np.uint32), oam.view(np.uint32))
        assert np.array_equal(av[tb].cpu().numpy().view(np.uint32), oav.view(np.uint32))
        assert int(step.item()) == 3 and opt.status() == 0
    finally:
        _cleanup()


def test_q4_tensor_beyond_2e31_elements():
    """One fp32 tensor of 2^31 + 4097 elements with 4-bit m and v (bf16 grads): whole
    128-element blocks across element 2^31, at both ends and at random, plus the
    1-element last block (a lone low nibble), bit-exact over 3 steps."""
    from oracle import q4 as O4
    n = (1 << 31) + 4097
    if _free_gib() < 25:
        pytest.skip("needs ~20 GiB of free device memory")
    from adamw_optimizer_step_tensor_gb300 import FusedAdamW
    try:
        rng = np.random.default_rng(66)
        nb = (n + 127) // 128
        w_p = synth.normal(n, 0.02, 67, "cuda")
        w_g = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        cm = torch.zeros((n + 1) // 2, dtype=torch.uint8, device="cuda")
        cv = torch.zeros((n + 1) // 2, dtype=torch.uint8, device="cuda")
        am, av = torch.zeros(nb, device="cuda"), torch.zeros(nb, device="cuda")
        opt = FusedAdamW([w_p], [w_g], [cm], [cv], [OA.f32(0.01)], mode="q4",
                         absmax_m=[am], absmax_v=[av])
        bidx, idx = _blocks_beyond_2e31(n, 128, rng)
        tb = torch.from_numpy(bidx).cuda()
        byte_idx = np.unique(idx // 2)   # whole blocks are 64 bytes; the last byte holds one code
        p = _take(w_p, idx).cpu().numpy()
        pm, pv = _take(cm, byte_idx).cpu().numpy(), _take(cv, byte_idx).cpu().numpy()
        oam, oav = am[tb].cpu().numpy(), av[tb].cpu().numpy()
        maps = O4.Maps4()
        lr, step = torch.tensor([OA.f32(1e-3)], device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
        for s in range(3):
            w_g.copy_(synth.normal(n, 1e-3, 68 + s, "cuda", torch.bfloat16))
            g = _take(w_g, idx).float().cpu().numpy()
            opt.step(lr, step)
            O4.step_f32(p, g, pm, pv, oam, oav, lr=OA.f32(1e-3), beta1=OA.f32(0.9),
                        beta2=OA.f32(0.999), eps=OA.f32(1e-8), wd=OA.f32(0.01), t=s + 1, maps=maps)
        torch.cuda.synchronize()
        assert np.array_equal(_take(w_p, idx).cpu().numpy().view(np.uint32), p.view(np.uint32))
        assert np.array_equal(_take(cm, byte_idx).cpu().numpy(), pm)
        assert np.array_equal(_take(cv, byte_idx).cpu().numpy(), pv)
        assert np.array_equal(am[tb].cpu().numpy().view(np.uint32), oam.view(np.uint32))
        assert np.array_equal(av[tb].cpu().numpy().view(np.uint32), oav.view(np.uint32))
        assert int(step.item()) == 3 and opt.status() == 0
    finally:
        _cleanup()


def _elementwise_full_size(w, step_fn, make_orc, check, n_steps, seed):
    """Shared driver for the GPT-2-list variants: sampled windows of every tensor."""
    rng = np.random.default_rng(seed)
    idx = _windows([p.numel() for p in w.ps], rng)
    orc = make_orc(idx)
    for s in range(n_steps):
        gs = w.step_grads(s)
        for k, g in enumerate(gs):
            g.copy_(synth.normal(g.numel(), 1e-3, synth.grad_seed(seed, s, k), "cuda"))
        for o, g, i in zip(orc, gs, idx):
            o.g = _take(g, i).cpu().numpy()
        w.step(s)
        step_fn(orc, float(w.lr_table[s % 100].item()), s)
    torch.cuda.synchronize()
    check(orc, idx)
    assert int(w.step_dev.item()) == n_steps
    assert w.status() == 0


def test_lion_gpt2_full_size_sampled():
    """The GPT-2-small list stepped with Lion (1-state plan, no exp_avg_sq), 10 steps."""
    from oracle import lion as OL
    w = bench.LionGpt2()
    try:
        def make(idx):
            return [OL.Tensor(p=_take(p, i).cpu().numpy(), g=None, m=_take(m, i).cpu().numpy(), wd=s.wd)
                    for p, m, i, s in zip(w.ps, w.ms, idx, w.specs)]

        def step(orc, lr, s):
            OL.step_f32(orc, lr=lr, beta1=OA.f32(0.9), beta2=OA.f32(0.99))

        def check(orc, idx):
            for k, (p, m, i, o) in enumerate(zip(w.ps, w.ms, idx, orc)):
                assert np.array_equal(_take(p, i).cpu().numpy().view(np.uint32), o.p.view(np.uint32)), k
                assert np.array_equal(_take(m, i).cpu().numpy().view(np.uint32), o.m.view(np.uint32)), k
        _elementwise_full_size(w, step, make, check, 10, 31)
    finally:
        del w
        _cleanup()


@pytest.mark.parametrize("rule", ["momentum", "rmsprop", "adagrad"])
def test_coupled_gpt2_full_size_sampled(rule):
    """The GPT-2-small list stepped with a coupled-L2 rule, 5 steps."""
    from oracle import coupled as OC
    w = bench.CoupledGpt2(rule)
    try:
        def make(idx):
            return [OC.Tensor(p=_take(p, i).cpu().numpy(), g=None, s=_take(m, i).cpu().numpy(), wd=s.wd)
                    for p, m, i, s in zip(w.ps, w.ms, idx, w.specs)]

        def step(orc, lr, s):
            OC.step_f32(orc, rule=rule, lr=lr, beta=OA.f32(0.9), eps=OA.f32(1e-8))

        def check(orc, idx):
            for k, (p, m, i, o) in enumerate(zip(w.ps, w.ms, idx, orc)):
                assert np.array_equal(_take(p, i).cpu().numpy().view(np.uint32), o.p.view(np.uint32)), k
                assert np.array_equal(_take(m, i).cpu().numpy().view(np.uint32), o.s.view(np.uint32)), k
        _elementwise_full_size(w, step, make, check, 5, 32)
    finally:
        del w
        _cleanup()


def test_q4_full_size_2e30_sampled_blocks():
    """One 2^30 fp32 tensor, 4-bit m and v, bf16 grads, lr 1e-3, wd 0.01, 10 steps."""
    from oracle import q4 as O4
    if _free_gib() < 10:
        pytest.skip("needs ~8 GiB of free device memory")
    w = bench.Q4()
    try:
        rng = np.random.default_rng(33)
        n = w.n_params
        blocks = np.unique(np.concatenate([[0, 1, n // 128 - 1], rng.integers(0, n // 128, 64)]))
        idx = (blocks[:, None] * 128 + np.arange(128)[None, :]).ravel()
        bidx = torch.from_numpy(blocks).cuda()
        byte_idx = (blocks[:, None] * 64 + np.arange(64)[None, :]).ravel()
        p = _take(w.p, idx).cpu().numpy()
        pm = _take(w.cm, byte_idx).cpu().numpy()
        pv = _take(w.cv, byte_idx).cpu().numpy()
        am = w.am[bidx].cpu().numpy()
        av = w.av[bidx].cpu().numpy()
        maps = O4.Maps4()
        gap = 0
        for s in range(10):
            w.g.copy_(synth.normal(n, 1e-3, synth.grad_seed(10, s), "cuda", torch.bfloat16))
            g = _take(w.g, idx).float().cpu().numpy()
            w.step(s)
            sc = OA.f32_scalars(lr=OA.f32(1e-3), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                                eps=OA.f32(1e-8), t=s + 1)
            _, m1, v1 = OA.elementwise_f32(p, g, O4.dequantize(pm, am, maps.smap, idx.size),
                                           O4.dequantize(pv, av, maps.umap, idx.size), sc,
                                           OA.decay_f32(sc.lr, OA.f32(0.01)))
            O4.step_f32(p, g, pm, pv, am, av, lr=OA.f32(1e-3), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                        eps=OA.f32(1e-8), wd=OA.f32(0.01), t=s + 1, maps=maps)
            torch.cuda.synchronize()
            kcm = O4.unpack(_take(w.cm, byte_idx).cpu().numpy(), idx.size)
            kcv = O4.unpack(_take(w.cv, byte_idx).cpu().numpy(), idx.size)
            gap += _division_rule_gap(kcm, m1, am, 128, maps.smap, maps.sthr)
            gap += _division_rule_gap(kcv, v1, av, 128, maps.umap, maps.uthr)
        print(f"4-bit codes that differ from the division rule: {gap} of {2 * 10 * idx.size}")
        assert gap <= 1e-3 * 2 * 10 * idx.size
        assert np.array_equal(_take(w.p, idx).cpu().numpy().view(np.uint32), p.view(np.uint32))
        assert np.array_equal(_take(w.cm, byte_idx).cpu().numpy(), pm)
        assert np.array_equal(_take(w.cv, byte_idx).cpu().numpy(), pv)
        assert np.array_equal(w.am[bidx].cpu().numpy().view(np.uint32), am.view(np.uint32))
        assert np.array_equal(w.av[bidx].cpu().numpy().view(np.uint32), av.view(np.uint32))
        assert int(w.step_dev.item()) == 10
    finally:
        del w
        _cleanup()


def test_adam_mini_llama3_full_size_sampled_blocks():
    """Adam-mini on the Llama-3-8B list (v per element / head / tensor), 3 steps: whole
    blocks sampled -- two query heads and one key head of layer 0, the whole wv of
    layer 31, two norm tensors -- plus windows of the per-element embedding and output."""
    from oracle import mini as OM
    if _free_gib() < 95:
        pytest.skip("needs ~90 GiB of free device memory")
    w = bench.MiniLlama3()
    try:
        hs, rs, gs, ms, vs = w._views
        blocks = synth.adam_mini_blocks(w.specs, dim=4096, n_heads=32)
        names = [s.name for s in w.specs]
        rng = np.random.default_rng(34)
        picks = []   # (tensor index, element indices, block length, v indices)
        for name, heads in (("layers.0.attention.wq", (0, 31)), ("layers.0.attention.wk", (5,))):
            k = names.index(name)
            for h in heads:
                picks.append((k, np.arange(h * blocks[k], (h + 1) * blocks[k]), blocks[k], np.array([h])))
        for name in ("layers.31.attention.wv", "layers.3.ffn_norm", "norm"):
            k = names.index(name)
            picks.append((k, np.arange(hs[k].numel()), blocks[k], np.array([0])))
        for name in ("tok_embeddings", "output"):
            k = names.index(name)
            i = _windows([hs[k].numel()], rng, n_rand=8)[0]
            picks.append((k, i, 1, i))
        orc = []
        for k, i, b, vi in picks:
            hi = _take(hs[k].view(torch.int16), i).cpu().numpy().view(np.uint16)
            orc.append(OM.Tensor(p=OR.join(hi, _take(rs[k], i).cpu().numpy()), g=None,
                                 m=_take(ms[k], i).cpu().numpy(), v=_take(vs[k], vi).cpu().numpy(),
                                 wd=0.0 if "norm" in names[k] else OA.f32(0.1), block=b))
        for s in range(3):
            for k, g in enumerate(gs):
                g.copy_(synth.normal(g.numel(), 1e-4, synth.grad_seed(11, s, k), "cuda", torch.bfloat16))
            for o, (k, i, b, vi) in zip(orc, picks):
                o.g = _take(gs[k], i).float().cpu().numpy()
            w.step(s)
            OM.step_f32(orc, lr=OA.f32(3e-4), beta1=OA.f32(0.9), beta2=OA.f32(0.999), eps=OA.f32(1e-8),
                        t=s + 1)
        torch.cuda.synchronize()
        for o, (k, i, b, vi) in zip(orc, picks):
            v = _take(vs[k], vi).cpu().numpy()
            ulps = np.abs(v.view(np.int32).astype(np.int64) - o.v.view(np.int32).astype(np.int64))
            assert ulps.max() <= 3, (names[k], int(ulps.max()))
            assert np.array_equal(_take(ms[k], i).cpu().numpy().view(np.uint32), o.m.view(np.uint32)), names[k]
            ohi, orem = OR.split(o.p)
            got = OR.join(_take(hs[k].view(torch.int16), i).cpu().numpy().view(np.uint16),
                          _take(rs[k], i).cpu().numpy())
            if b == 1:
                assert np.array_equal(got.view(np.uint32), o.p.view(np.uint32)), names[k]
            else:
                assert np.all(np.abs(got.astype(np.float64) - o.p) <= 2.0 ** -21 * (np.abs(o.p) + 1e-6)), names[k]
        assert int(w.step_dev.item()) == 3
        assert w.opt.status() == 0
    finally:
        del w
        _cleanup()
