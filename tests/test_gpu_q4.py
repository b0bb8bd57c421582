"""GPU parity: AdamW with 4-bit blockwise-quantised moments (mode "q4").

Params, packed codes and per-block absmax are bit-exact against the
strict-fp32 4-bit oracle on ragged tensor lists (odd sizes leave a lone low
nibble, partial and empty half-warp blocks, a misaligned tensor on the
element path) for fp32/fp16/bf16 grads; the first step from zero state also
matches the closed form of "Fix decoupled weight decay ordering in the CUDA
Adam/AdEMAMix kernels" (bitsandbytes PR #2040); the AMP skip leaves
everything as it was.
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW
from oracle import adamw as OA
from oracle import q4 as O4
from oracle import q8 as OQ

from _support import (assert_guards_intact, assert_max_abs, assert_single_step_rel,
                      assert_state_bitexact, bits_equal, dev, empty, first_mismatch, grads_of, host,
                      scalar_f32, scalar_i32, to_dev, zeros)

pytestmark = pytest.mark.gpu
f32 = OA.f32
B1, B2, EPS = f32(0.9), f32(0.999), f32(1e-8)
SIZES = [1, 7, 127, 128, 129, 255, 256, 257, 2048 + 100, 8192 + 301, 70001, 0]


def _view(a, misalign):
    if not misalign:
        return dev(a)
    return dev(a, shift=1)   # one element off the 16-byte grid, guard bands on both sides


def _build(sizes, gdtype, seed, zero_state, misalign=False):
    rng = np.random.default_rng(seed)
    st = []
    for n in sizes:
        nb = OQ.n_blocks(n, O4.BLOCK)
        p = rng.normal(0, 0.02, n).astype(np.float32)
        pm = O4.pack(rng.integers(0, 16, n).astype(np.uint8))
        pv = O4.pack(rng.integers(0, 16, n).astype(np.uint8))
        am = np.zeros(nb, np.float32) if zero_state else rng.uniform(0, 1e-3, nb).astype(np.float32)
        av = np.zeros(nb, np.float32) if zero_state else rng.uniform(0, 1e-6, nb).astype(np.float32)
        st.append(dict(p=p, cm=pm, cv=pv, am=am, av=av))
    d = [{k: (_view(v, misalign) if k == "p" else dev(v)) for k, v in s.items()} for s in st]
    gs = [empty(n, gdtype) for n in sizes]
    opt = FusedAdamW([x["p"] for x in d], gs, [x["cm"] for x in d], [x["cv"] for x in d],
                     [f32(0.01) if i % 2 else 0.0 for i in range(len(sizes))], mode="q4",
                     absmax_m=[x["am"] for x in d], absmax_v=[x["av"] for x in d])
    return opt, st, d, gs, rng


def _steps(opt, st, d, gs, rng, gdtype, n_steps, lr=1e-3, scale=None):
    """n_steps against the oracle; ``scale``: grads scaled by it and the loss
    scale passed to both sides (the scaled kernel instantiation)."""
    maps = O4.Maps4()
    lr_d, step = scalar_f32(f32(lr)), scalar_i32(0)
    scale_d = None if scale is None else scalar_f32(f32(scale))
    for t in range(1, n_steps + 1):
        wide = []
        for g in gs:
            x = rng.normal(0, 1e-3, g.numel()) * (1.0 if scale is None else scale)
            tg, w = grads_of(x.astype(np.float32), gdtype)
            g.copy_(tg)
            wide.append(w)
        opt.step(lr_d, step, betas=(B1, B2), eps=EPS, grad_scale=scale_d)
        for i, (s, w) in enumerate(zip(st, wide)):
            O4.step_f32(s["p"], w, s["cm"], s["cv"], s["am"], s["av"], lr=f32(lr), beta1=B1,
                        beta2=B2, eps=EPS, wd=f32(0.01) if i % 2 else 0.0, t=t, maps=maps,
                        grad_scale=None if scale is None else f32(scale))
        torch.cuda.synchronize()
        assert_guards_intact()
        for i, (s, x) in enumerate(zip(st, d)):
            assert bits_equal(host(x["p"]), s["p"]), f"t{t} tensor {i} p: {first_mismatch(host(x['p']), s['p'])}"
            assert np.array_equal(host(x["cm"]), s["cm"]), f"t{t} tensor {i} m codes"
            assert np.array_equal(host(x["cv"]), s["cv"]), f"t{t} tensor {i} v codes"
            assert bits_equal(host(x["am"]), s["am"]), f"t{t} tensor {i} absmax m"
            assert bits_equal(host(x["av"]), s["av"]), f"t{t} tensor {i} absmax v"
    assert int(step.item()) == n_steps


@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32, torch.float16])
def test_q4_steps_bitexact(gdtype):
    opt, st, d, gs, rng = _build(SIZES, gdtype, seed=31, zero_state=False)
    _steps(opt, st, d, gs, rng, gdtype, 4)


@pytest.mark.parametrize("gdtype", [torch.float16, torch.bfloat16, torch.float32])
def test_q4_steps_bitexact_with_a_loss_scale(gdtype):
    """A loss scale of 3000 (its reciprocal rounds) on every step: the scaled
    kernel instantiation, bit-exact."""
    opt, st, d, gs, rng = _build(SIZES, gdtype, seed=37, zero_state=False)
    _steps(opt, st, d, gs, rng, gdtype, 3, scale=3000.0)


def test_q4_from_zero_state_bitexact():
    opt, st, d, gs, rng = _build(SIZES, torch.bfloat16, seed=32, zero_state=True)
    _steps(opt, st, d, gs, rng, torch.bfloat16, 3, lr=1e-2)


def test_q4_element_path_on_misaligned_params():
    opt, st, d, gs, rng = _build([1, 129, 1000, 4099], torch.float32, seed=33, zero_state=False,
                                 misalign=True)
    _steps(opt, st, d, gs, rng, torch.float32, 2)


def test_q4_first_step_closed_form():
    n = 100_001
    opt, st, d, gs, rng = _build([n], torch.float32, seed=34, zero_state=True)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    gs[0].copy_(dev(g))
    p0 = st[0]["p"].astype(np.float64)
    opt.step(scalar_f32(f32(0.1)), scalar_i32(0), betas=(B1, B2), eps=EPS)
    torch.cuda.synchronize()
    lr = f32(0.1)
    want = p0 - lr * g / (np.abs(g) + EPS)           # tensor 0 has wd 0
    got = host(d[0]["p"]).astype(np.float64)
    assert np.max(np.abs(got - want) / (np.abs(want) + lr)) < 8 * 2.0 ** -24
    assert host(d[0]["cm"])[-1] >> 4 == 0             # odd n: the last high nibble stays 0


def test_q4_amp_skip_leaves_codes_and_absmax():
    n = 3001
    opt, st, d, gs, rng = _build([n], torch.float16, seed=35, zero_state=False)
    gs[0].copy_(dev((rng.normal(0, 1e-3, n) * 1024).astype(np.float16)))
    gs[0][5] = float("nan")
    before = {k: host(v) for k, v in d[0].items()}
    found, step = scalar_f32(0.0), scalar_i32(7)
    opt.check_nonfinite(found)
    opt.step(scalar_f32(1e-3), step, grad_scale=scalar_f32(1024.0), found_inf=found)
    torch.cuda.synchronize()
    for k, v in d[0].items():
        assert np.array_equal(host(v).view(np.uint8), before[k].view(np.uint8)), k
    assert int(step.item()) == 7


def test_q4_export_import_match_oracle():
    from adamw_optimizer_step_tensor_gb300 import _capi as C
    from oracle import qmap
    n = 10_001
    opt, st, d, gs, rng = _build([n], torch.bfloat16, seed=36, zero_state=False)
    maps = O4.Maps4()
    x = (rng.normal(0, 1e-3, n) * rng.uniform(0, 1, n)).astype(np.float32)
    x[:128] = 0.0                        # an all-zero block
    x[300] = np.nan                      # NaN poisons its block's absmax and codes 0
    nb = OQ.n_blocks(n, O4.BLOCK)
    sh = torch.cuda.current_stream().cuda_stream
    for which, table, thr in ((0, maps.smap, maps.sthr), (1, maps.umap, maps.uthr)):
        xs = x if which == 0 else np.abs(x)
        xd = dev(xs)
        codes = empty((n + 1) // 2, torch.uint8)
        am = empty(nb, torch.float32)
        C.adamw_q4_quant(opt.plan, which, xd.data_ptr(), codes.data_ptr(), am.data_ptr(), n, sh)
        out = empty(n, torch.float32)
        C.adamw_q4_dequant(opt.plan, which, codes.data_ptr(), am.data_ptr(), out.data_ptr(), n, sh)
        torch.cuda.synchronize()
        oc, oa = O4.quantize_blockwise(xs, table, thr)
        assert np.array_equal(host(codes), O4.pack(oc)), which
        assert bits_equal(host(am), oa), which
        assert np.array_equal(host(out), OQ.dequantize(oc, oa, table, O4.BLOCK), equal_nan=True), which
    assert qmap.empty_block_code(maps.umap) == 0
    with pytest.raises(C.AdamWError):   # an 8-bit plan refuses the 4-bit calls
        opt8 = FusedAdamW([d[0]["p"]], [gs[0]], [zeros(n, torch.uint8)],
                          [zeros(n, torch.uint8)], [0.0], mode="q8",
                          absmax_m=[zeros(OQ.n_blocks(n))],
                          absmax_v=[zeros(OQ.n_blocks(n))])
        C.adamw_q4_dequant(opt8.plan, 0, codes.data_ptr(), am.data_ptr(), out.data_ptr(), n, sh)


def _same_or_both_nan(a, b):
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    nan = np.isnan(a)
    return np.array_equal(nan, np.isnan(b)) and bits_equal(a[~nan], b[~nan])


def test_q4_nonfinite_grads_without_skip_match_oracle():
    """A step that is not skipped on non-finite grads (no found_inf given):
    NaN and +-inf reach the moments, the block absmax (a maximum over float
    bits, so a NaN wins) and the nearest-code searches of both maps, whose
    NaN inputs take code 0.  Codes bit-exact, params and absmax equal up to
    NaN payloads (the CPU and the GPU make different default NaNs)."""
    n = 1000
    opt, st, d, gs, rng = _build([n], torch.float32, seed=37, zero_state=False)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    g[5], g[300], g[700], g[701] = np.nan, np.inf, -np.inf, np.inf
    gs[0].copy_(dev(g))
    opt.step(scalar_f32(f32(1e-3)), scalar_i32(0), betas=(B1, B2), eps=EPS)
    s = st[0]
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        O4.step_f32(s["p"], g, s["cm"], s["cv"], s["am"], s["av"], lr=f32(1e-3), beta1=B1,
                    beta2=B2, eps=EPS, wd=0.0, t=1, maps=O4.Maps4())
    torch.cuda.synchronize()
    x = d[0]
    assert np.array_equal(host(x["cm"]), s["cm"])
    assert np.array_equal(host(x["cv"]), s["cv"])
    for k in ("p", "am", "av"):
        assert _same_or_both_nan(host(x[k]), s[k]), k
    assert np.isnan(host(x["am"])[0]) and np.isinf(host(x["av"])[2])
