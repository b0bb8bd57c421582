"""GPU parity: AdamW with 8-bit blockwise-quantised moments.

Params, codes and per-block absmax are bit-exact against the strict-fp32
oracle (the discrete outputs are defined against that mode); the first step
from zero state also matches the closed form of "Fix decoupled weight decay
ordering in the CUDA Adam/AdEMAMix kernels" (bitsandbytes PR #2040).  User
maps dense enough to need 2 and 4 threshold compares per lookup, and
non-finite grads on a step that is not skipped, stay bit-exact too.
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi as C
from oracle import adamw as OA
from oracle import q8 as OQ

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu
f32 = OA.f32
B1, B2, EPS = f32(0.9), f32(0.999), f32(1e-8)
SIZES = [1, 255, 256, 257, 2048 + 100, 8192 + 300, 70001, 0]


def _view(a, misalign):
    if not misalign:
        return dev(a)
    return dev(a, shift=1)   # one element off the 16-byte grid, guard bands on both sides


def _build(sizes, gdtype, seed, zero_state, misalign=False):
    rng = np.random.default_rng(seed)
    st = []
    for n in sizes:
        nb = OQ.n_blocks(n)
        p = rng.normal(0, 0.02, n).astype(np.float32)
        cm = rng.integers(0, 256, n).astype(np.uint8)
        cv = rng.integers(0, 256, n).astype(np.uint8)
        am = np.zeros(nb, np.float32) if zero_state else rng.uniform(0, 1e-3, nb).astype(np.float32)
        av = np.zeros(nb, np.float32) if zero_state else rng.uniform(0, 1e-6, nb).astype(np.float32)
        st.append(dict(p=p, cm=cm, cv=cv, am=am, av=av))
    d = [{k: (_view(v, misalign) if k == "p" else dev(v)) for k, v in s.items()} for s in st]
    gs = [empty(n, gdtype) for n in sizes]
    opt = FusedAdamW([x["p"] for x in d], gs, [x["cm"] for x in d], [x["cv"] for x in d],
                     [f32(0.01)] * len(sizes), mode="q8", absmax_m=[x["am"] for x in d],
                     absmax_v=[x["av"] for x in d])
    return opt, st, d, gs, rng


@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32, torch.float16])
def test_q8_steps_bitexact(gdtype):
    opt, st, d, gs, rng = _build(SIZES, gdtype, seed=11, zero_state=False)
    maps = OQ.Maps()
    lr, step = scalar_f32(f32(1e-3)), scalar_i32(0)
    for t in range(1, 5):
        wide = []
        for g in gs:
            tg, w = grads_of(rng.normal(0, 1e-3, g.numel()).astype(np.float32), gdtype)
            g.copy_(tg)
            wide.append(w)
        opt.step(lr, step, betas=(B1, B2), eps=EPS)
        for s, w in zip(st, wide):
            OQ.step_f32(s["p"], w, s["cm"], s["cv"], s["am"], s["av"], lr=f32(1e-3), beta1=B1,
                        beta2=B2, eps=EPS, wd=f32(0.01), t=t, maps=maps)
        torch.cuda.synchronize()
        assert_guards_intact()
        for i, (s, x) in enumerate(zip(st, d)):
            assert bits_equal(host(x["p"]), s["p"]), f"t{t} tensor {i} p: {first_mismatch(host(x['p']), s['p'])}"
            assert np.array_equal(host(x["cm"]), s["cm"]), f"t{t} tensor {i} m codes"
            assert np.array_equal(host(x["cv"]), s["cv"]), f"t{t} tensor {i} v codes"
            assert bits_equal(host(x["am"]), s["am"]), f"t{t} tensor {i} absmax m"
            assert bits_equal(host(x["av"]), s["av"]), f"t{t} tensor {i} absmax v"


@pytest.mark.parametrize("gdtype", [torch.float16, torch.bfloat16, torch.float32])
def test_q8_steps_bitexact_with_a_loss_scale(gdtype):
    """A loss scale of 3000 (its reciprocal rounds) on every step: the scaled
    kernel instantiation, bit-exact on the ragged list."""
    opt, st, d, gs, rng = _build(SIZES, gdtype, seed=17, zero_state=False)
    maps = OQ.Maps()
    lr, step, scale = scalar_f32(f32(1e-3)), scalar_i32(0), scalar_f32(f32(3000.0))
    for t in range(1, 4):
        wide = []
        for g in gs:
            tg, w = grads_of((rng.normal(0, 1e-3, g.numel()) * 3000.0).astype(np.float32), gdtype)
            g.copy_(tg)
            wide.append(w)
        opt.step(lr, step, betas=(B1, B2), eps=EPS, grad_scale=scale)
        for s, w in zip(st, wide):
            OQ.step_f32(s["p"], w, s["cm"], s["cv"], s["am"], s["av"], lr=f32(1e-3), beta1=B1,
                        beta2=B2, eps=EPS, wd=f32(0.01), t=t, maps=maps, grad_scale=f32(3000.0))
        torch.cuda.synchronize()
        assert_guards_intact()
        for i, (s, x) in enumerate(zip(st, d)):
            assert bits_equal(host(x["p"]), s["p"]), f"t{t} tensor {i} p: {first_mismatch(host(x['p']), s['p'])}"
            assert np.array_equal(host(x["cm"]), s["cm"]), f"t{t} tensor {i} m codes"
            assert np.array_equal(host(x["cv"]), s["cv"]), f"t{t} tensor {i} v codes"
            assert bits_equal(host(x["am"]), s["am"]), f"t{t} tensor {i} absmax m"
            assert bits_equal(host(x["av"]), s["av"]), f"t{t} tensor {i} absmax v"
    assert int(step.item()) == 3


def test_q8_element_path_on_misaligned_params():
    """Params 4 bytes off the 16-byte grid: every block of those tensors takes
    the element path (scalar loads, per-element predicates), several warps of
    the 1024-thread CTA at once; still bit-exact."""
    opt, st, d, gs, rng = _build([1, 257, 1000, 9000], torch.float32, seed=20, zero_state=False,
                                 misalign=True)
    maps = OQ.Maps()
    lr, step = scalar_f32(f32(1e-3)), scalar_i32(0)
    for t in range(1, 3):
        wide = []
        for g in gs:
            tg, w = grads_of(rng.normal(0, 1e-3, g.numel()).astype(np.float32), torch.float32)
            g.copy_(tg)
            wide.append(w)
        opt.step(lr, step, betas=(B1, B2), eps=EPS)
        for s, w in zip(st, wide):
            OQ.step_f32(s["p"], w, s["cm"], s["cv"], s["am"], s["av"], lr=f32(1e-3), beta1=B1,
                        beta2=B2, eps=EPS, wd=f32(0.01), t=t, maps=maps)
        torch.cuda.synchronize()
        assert_guards_intact()
        for i, (s, x) in enumerate(zip(st, d)):
            assert bits_equal(host(x["p"]), s["p"]), f"t{t} tensor {i} p"
            assert np.array_equal(host(x["cm"]), s["cm"]), f"t{t} tensor {i} m codes"
            assert np.array_equal(host(x["cv"]), s["cv"]), f"t{t} tensor {i} v codes"
            assert bits_equal(host(x["am"]), s["am"]) and bits_equal(host(x["av"]), s["av"])


def test_q8_first_step_closed_form():
    n = 100_000
    opt, st, d, gs, rng = _build([n], torch.float32, seed=12, zero_state=True)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    gs[0].copy_(dev(g))
    p0 = st[0]["p"].astype(np.float64)
    opt.step(scalar_f32(f32(0.1)), scalar_i32(0), betas=(B1, B2), eps=EPS)
    torch.cuda.synchronize()
    lr, wd = f32(0.1), f32(0.01)
    want = p0 * (1 - lr * wd) - lr * g / (np.abs(g) + EPS)
    got = host(d[0]["p"]).astype(np.float64)
    assert np.max(np.abs(got - want) / (np.abs(want) + lr)) < 8 * 2.0 ** -24


def test_q8_export_import_match_oracle():
    n = 10_000
    opt, st, d, gs, rng = _build([n], torch.bfloat16, seed=13, zero_state=False)
    maps = OQ.Maps()
    x = (rng.normal(0, 1e-3, n) * rng.uniform(0, 1, n)).astype(np.float32)
    x[:256] = 0.0                       # an all-zero block
    x[300] = np.nan                     # NaN poisons its block's absmax and codes 0
    xd = dev(x)
    nb = OQ.n_blocks(n)
    for which, table, thr in ((0, maps.smap, maps.sthr), (1, maps.umap, maps.uthr)):
        xs = x if which == 0 else np.abs(x)
        xd.copy_(dev(xs))
        codes = empty(n, torch.uint8)
        am = empty(nb, torch.float32)
        sh = torch.cuda.current_stream().cuda_stream
        C.adamw_q8_quant(opt.plan, which, xd.data_ptr(), codes.data_ptr(), am.data_ptr(), n, sh)
        out = empty(n, torch.float32)
        C.adamw_q8_dequant(opt.plan, which, codes.data_ptr(), am.data_ptr(), out.data_ptr(), n, sh)
        torch.cuda.synchronize()
        oc, oa = OQ.quantize_blockwise(xs, table, thr)
        assert np.array_equal(host(codes), oc)
        assert bits_equal(host(am), oa)
        # the NaN block dequantises to NaN (payloads may differ between CPU and GPU)
        assert np.array_equal(host(out), OQ.dequantize(oc, oa, table), equal_nan=True)


def test_q8_custom_maps_through_set_maps():
    """A user map (uniform 256 levels) replaces the default; parity still bit-exact."""
    n = 5000
    opt, st, d, gs, rng = _build([n], torch.bfloat16, seed=14, zero_state=False)
    smap = np.unique(np.concatenate([np.linspace(-1, 1, 255), [0.999]]).astype(np.float32))
    assert smap.size == 256 and 0.0 in smap
    umap = np.linspace(0, 1, 256).astype(np.float32)
    opt.set_maps(smap, umap)
    maps = OQ.Maps(smap, umap)
    tg, w = grads_of(rng.normal(0, 1e-3, n).astype(np.float32), torch.bfloat16)
    gs[0].copy_(tg)
    opt.step(scalar_f32(f32(1e-3)), scalar_i32(2), betas=(B1, B2), eps=EPS)
    s = st[0]
    OQ.step_f32(s["p"], w, s["cm"], s["cv"], s["am"], s["av"], lr=f32(1e-3), beta1=B1, beta2=B2,
                eps=EPS, wd=f32(0.01), t=3, maps=maps)
    torch.cuda.synchronize()
    assert bits_equal(host(d[0]["p"]), s["p"])
    assert np.array_equal(host(d[0]["cm"]), s["cm"])
    assert np.array_equal(host(d[0]["cv"]), s["cv"])


def test_q8_rejects_maps_without_zero():
    n = 300
    opt, st, d, gs, rng = _build([n], torch.bfloat16, seed=15, zero_state=True)
    bad = np.linspace(-1, 1, 256).astype(np.float32)   # even count: 0 is not a level
    assert 0.0 not in bad
    with pytest.raises(C.AdamWError):
        opt.set_maps(bad, np.linspace(0, 1, 256).astype(np.float32))


def test_q8_amp_skip_leaves_codes_and_absmax():
    n = 3000
    opt, st, d, gs, rng = _build([n], torch.float16, seed=16, zero_state=False)
    gs[0].copy_(dev((rng.normal(0, 1e-3, n) * 1024).astype(np.float16)))
    gs[0][5] = float("inf")
    before = {k: host(v) for k, v in d[0].items()}
    found, step = scalar_f32(0.0), scalar_i32(7)
    opt.check_nonfinite(found)
    opt.step(scalar_f32(1e-3), step, grad_scale=scalar_f32(1024.0), found_inf=found)
    torch.cuda.synchronize()
    for k, v in d[0].items():
        assert np.array_equal(host(v).view(np.uint8), before[k].view(np.uint8)), k
    assert int(step.item()) == 7


def _cluster_map(k):
    """A signed map with k extra levels 0.0008 apart just above 0.6, where a
    bucket of the nearest-code search is 2^-8 wide: its thresholds crowd
    into one bucket, so the search must compare more of them (the plan's
    refine count: 2 for k = 3, 3 for k = 5, 5 for k = 7)."""
    grid = np.linspace(-1, 1, 241)
    cluster = 0.6 + 0.0008 * np.arange(1, k + 1)
    n_pad = 256 - grid.size - k
    pads = (grid[12:12 + n_pad] + grid[13:13 + n_pad]) / 2
    m = np.sort(np.concatenate([grid, cluster, pads])).astype(np.float32)
    assert m.size == 256 and np.unique(m).size == 256 and 0.0 in m
    return m


@pytest.mark.parametrize("k", [3, 5])
def test_q8_dense_maps_take_more_compares(k):
    """Maps whose thresholds crowd a bucket run the kernel variants with 2 and
    4 threshold compares per lookup; codes, absmax and params stay bit-exact."""
    n = 60_000
    opt, st, d, gs, rng = _build([n], torch.bfloat16, seed=17, zero_state=False)
    smap = _cluster_map(k)
    umap = np.linspace(0, 1, 256).astype(np.float32)
    opt.set_maps(smap, umap)
    maps = OQ.Maps(smap, umap)
    lr, step = scalar_f32(f32(1e-3)), scalar_i32(0)
    s, x = st[0], d[0]
    in_cluster = 0
    for t in range(1, 3):
        tg, w = grads_of(rng.normal(0, 1e-3, n).astype(np.float32), torch.bfloat16)
        gs[0].copy_(tg)
        opt.step(lr, step, betas=(B1, B2), eps=EPS)
        OQ.step_f32(s["p"], w, s["cm"], s["cv"], s["am"], s["av"], lr=f32(1e-3), beta1=B1,
                    beta2=B2, eps=EPS, wd=f32(0.01), t=t, maps=maps)
        torch.cuda.synchronize()
        assert bits_equal(host(x["p"]), s["p"]), f"t{t} p: {first_mismatch(host(x['p']), s['p'])}"
        assert np.array_equal(host(x["cm"]), s["cm"]), f"t{t} m codes"
        assert np.array_equal(host(x["cv"]), s["cv"]), f"t{t} v codes"
        assert bits_equal(host(x["am"]), s["am"]) and bits_equal(host(x["av"]), s["av"]), f"t{t}"
        in_cluster += int(np.sum((smap[s["cm"]] > 0.6) & (smap[s["cm"]] < 0.607)))
    assert in_cluster > 100        # the crowded bucket was exercised


def test_q8_maps_too_dense_for_the_search_are_refused():
    n = 300
    opt, st, d, gs, rng = _build([n], torch.bfloat16, seed=18, zero_state=True)
    with pytest.raises(C.AdamWError, match="too dense"):
        opt.set_maps(_cluster_map(7), np.linspace(0, 1, 256).astype(np.float32))


def _same_or_both_nan(a, b):
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    nan = np.isnan(a)
    return np.array_equal(nan, np.isnan(b)) and bits_equal(a[~nan], b[~nan])


def test_q8_nonfinite_grads_without_skip_match_oracle():
    """A step that is not skipped on non-finite grads (no found_inf given):
    NaN and +-inf reach the moments, the block absmax (a maximum over float
    bits, so a NaN wins) and both nearest-code searches, whose NaN inputs
    take code 0.  Codes bit-exact, params and absmax equal up to NaN payloads
    (the CPU and the GPU make different default NaNs)."""
    n = 2000
    opt, st, d, gs, rng = _build([n], torch.float32, seed=19, zero_state=False)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    g[5], g[600], g[1400], g[1401] = np.nan, np.inf, -np.inf, np.inf
    gs[0].copy_(dev(g))
    opt.step(scalar_f32(f32(1e-3)), scalar_i32(0), betas=(B1, B2), eps=EPS)
    s = st[0]
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        OQ.step_f32(s["p"], g, s["cm"], s["cv"], s["am"], s["av"], lr=f32(1e-3), beta1=B1,
                    beta2=B2, eps=EPS, wd=f32(0.01), t=1, maps=OQ.Maps())
    torch.cuda.synchronize()
    x = d[0]
    assert np.array_equal(host(x["cm"]), s["cm"])
    assert np.array_equal(host(x["cv"]), s["cv"])
    for k in ("p", "am", "av"):
        assert _same_or_both_nan(host(x[k]), s[k]), k
    assert np.isnan(host(x["am"])[0]) and np.isinf(host(x["av"])[2])
