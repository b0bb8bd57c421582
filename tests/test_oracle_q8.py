"""Pins for the 8-bit code maps, the quantiser and the 8-bit-state step (CPU only).

The map contents are *parity unpinned* by the pages (they never print it);
pinned here are its structural invariants (256 distinct sorted values, exact 0
and 1.0, the per-decade counts of the dynamic-exponent layout), the
threshold quantiser against a brute-force nearest search, and the 8-bit step
against the first-step closed form of "Fix decoupled weight decay ordering in
the CUDA Adam/AdEMAMix kernels" (bitsandbytes PR #2040): a zero state
quantises exactly, so one step from it is ``p0*(1-lr*wd) - lr*g/(|g|+eps)``.
"""

import math

import numpy as np
import pytest

from oracle import adamw as A
from oracle import q8, qmap

F32 = np.float32


@pytest.fixture(scope="module")
def maps():
    return q8.Maps()


def test_map_structure(maps):
    for table, lo in ((maps.smap, -1.0), (maps.umap, 0.0)):
        assert table.dtype == F32 and table.size == 256
        assert np.all(np.diff(table.astype(np.float64)) > 0)
        assert table[-1] == 1.0 and 0.0 in table and table[0] >= lo
    # dynamic exponent layout: per decade [10**-(E+1), 10**-E) the counts halve
    pos_s = maps.smap[maps.smap > 0].astype(np.float64)
    pos_u = maps.umap[maps.umap > 0].astype(np.float64)
    for e in range(7):
        lo_, hi_ = 10.0 ** -(e + 1), 10.0 ** -e
        assert np.sum((pos_s >= lo_) & (pos_s < hi_)) == 2 ** (6 - e)
        assert np.sum((pos_u >= lo_) & (pos_u < hi_)) == 2 ** (7 - e)
    # signed map is symmetric apart from the extra +1.0
    neg = -maps.smap[maps.smap < 0][::-1]
    assert np.array_equal(neg, pos_s[:-1].astype(F32))
    assert qmap.zero_code(maps.smap) == 127 and qmap.zero_code(maps.umap) == 0


def test_map_values_are_the_rounded_rationals(maps):
    # spot values of the construction: top fraction bin at E=0, lowest at E=6
    assert maps.smap[-2] == F32(0.1 + 63.5 * 0.9 / 64)
    assert maps.smap[128] == F32(1e-6 * 0.55)
    assert maps.umap[1] == F32(1e-6 * (0.1 + 0.5 * 0.9 / 2))


def _probe_points(table, thr, rng):
    pts = [table, thr, np.nextafter(thr, F32(-np.inf)), np.nextafter(thr, F32(np.inf)),
           np.array([0.0, -0.0, 1.0, -1.0, 1e-30, -1e-30], F32)]
    mags = 10.0 ** rng.uniform(-9, 0, 3000)
    pts.append((mags * rng.choice([-1.0, 1.0], mags.size)).astype(F32))
    return np.concatenate([np.asarray(p, F32) for p in pts])


@pytest.mark.parametrize("which", ["smap", "umap"])
def test_threshold_quantiser_equals_bruteforce(maps, which):
    table = getattr(maps, which)
    thr = qmap.thresholds(table)
    x = _probe_points(table, thr, np.random.default_rng(4))
    assert np.array_equal(qmap.quantize(x, table, thr), qmap.quantize_bruteforce(x, table))


def test_map_values_quantise_to_themselves(maps):
    for table in (maps.smap, maps.umap):
        assert np.array_equal(qmap.quantize(table, table), np.arange(256))


def test_nan_quantises_to_code_zero(maps):
    assert qmap.quantize(np.array([np.nan], F32), maps.smap)[0] == 0
    assert qmap.quantize_bruteforce(np.array([np.nan], F32), maps.smap)[0] == 0


def test_blockwise_roundtrip_error_bound(maps):
    rng = np.random.default_rng(5)
    x = (rng.normal(0, 1e-3, 1000) * rng.uniform(0, 1, 1000)).astype(F32)
    codes, amax = q8.quantize_blockwise(x, maps.smap, maps.sthr)
    assert amax.size == 4  # 256 + 256 + 256 + 232
    for b in range(4):
        xb = x[b * 256:(b + 1) * 256]
        assert amax[b] == np.max(np.abs(xb))
    y = q8.dequantize(codes, amax, maps.smap)
    # nearest code: the error is at most half the gap to the neighbouring code,
    # or, past the most negative code, the distance from it to -1
    t = maps.smap.astype(np.float64)
    gap = np.maximum(np.diff(t, prepend=t[0])[codes], np.diff(t, append=t[-1])[codes])
    bound = np.maximum(0.5 * gap, np.where(codes == 0, 1.0 + t[0], 0.0))
    a = amax[np.arange(x.size) // 256].astype(np.float64)
    assert np.all(np.abs(y - x) <= bound * a * (1 + 1e-5) + 1e-12)


def test_exact_block_recovers_codes_and_absmax(maps):
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 256, 512).astype(np.uint8)
    codes[0] = 255          # +1.0 so the block max is exactly A
    codes[256] = 255
    A_ = np.array([2.0 ** -7, 2.0 ** -11], F32)  # powers of two: products exact
    x = q8.dequantize(codes, A_, maps.smap)
    c2, a2 = q8.quantize_blockwise(x, maps.smap, maps.sthr)
    assert np.array_equal(a2, A_) and np.array_equal(c2, codes)


def test_zero_block_is_zero_code_and_zero_absmax(maps):
    x = np.zeros(300, F32)
    x[5] = -0.0
    codes, amax = q8.quantize_blockwise(x, maps.smap, maps.sthr)
    assert np.all(amax == 0) and np.all(codes == 127)
    assert np.all(q8.dequantize(codes, amax, maps.smap) == 0)


def test_absmax_over_bits_equals_float_max():
    rng = np.random.default_rng(7)
    x = rng.normal(0, 1, 777).astype(F32)
    assert q8.absmax_bits(x) == np.max(np.abs(x))


def _closed_form(p, g, lr, wd, eps):
    return p * (1 - lr * wd) - lr * g / (np.abs(g) + eps)


def test_first_step_closed_form_q8(maps):
    rng = np.random.default_rng(8)
    n = 1000
    p = rng.normal(0, 0.02, n).astype(F32)
    g = rng.normal(0, 1e-3, n).astype(F32)
    hp = dict(lr=A.f32(0.1), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8),
              wd=A.f32(0.1), t=1)
    nb = q8.n_blocks(n)
    cm = rng.integers(0, 256, n).astype(np.uint8)   # any codes: absmax 0 means zero state
    cv = rng.integers(0, 256, n).astype(np.uint8)
    am, av = np.zeros(nb, F32), np.zeros(nb, F32)
    p32 = p.copy()
    q8.step_f32(p32, g, cm, cv, am, av, maps=maps, **hp)
    want = _closed_form(p.astype(np.float64), g.astype(np.float64), hp["lr"], hp["wd"], hp["eps"])
    assert np.max(np.abs(p32 - want) / (np.abs(want) + hp["lr"])) < 8 * 2.0 ** -24
    # and the float64 form of the same method
    p64, _, _ = q8.step_fp64(p, g, (np.zeros(n, np.uint8), np.zeros(nb, F32)),
                             (np.zeros(n, np.uint8), np.zeros(nb, F32)), maps=maps, **hp)
    assert np.allclose(p64, want, rtol=1e-13, atol=1e-16)
    # the new states are the quantised first moments (1-b1)g and (1-b2)g^2
    assert np.array_equal(am, np.array([q8.absmax_bits(F32(1 - F32(0.9)) * g[i * 256:(i + 1) * 256])
                                        for i in range(nb)], F32))


def test_q8_update_uses_unquantised_moments(maps):
    """p' equals the fp32-state step fed with the dequantised old state."""
    rng = np.random.default_rng(9)
    n = 512
    p = rng.normal(0, 0.02, n).astype(F32)
    g = rng.normal(0, 1e-3, n).astype(F32)
    cm = rng.integers(0, 256, n).astype(np.uint8)
    cv = rng.integers(0, 256, n).astype(np.uint8)
    am = np.array([1e-3, 2e-3], F32)
    av = np.array([1e-6, 3e-6], F32)
    m = q8.dequantize(cm, am, maps.smap)
    v = q8.dequantize(cv, av, maps.umap)
    hp = dict(lr=A.f32(1e-3), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8))
    x = A.Tensor(p=p.copy(), g=g, m=m.copy(), v=v.copy(), wd=A.f32(0.01))
    A.step_f32([x], t=5, **hp)
    p8 = p.copy()
    q8.step_f32(p8, g, cm, cv, am, av, wd=A.f32(0.01), t=5, maps=maps, **hp)
    assert np.array_equal(p8, x.p)
    assert np.array_equal(q8.quantize_blockwise(x.m, maps.smap, maps.sthr)[0], cm)


def test_q8_state_error_order_of_page_figure(maps):
    """Quantised vs fp32 moments drift apart by ~1e-3 relative per step (page: 6.6e-4)."""
    rng = np.random.default_rng(10)
    n = 4096
    p = rng.normal(0, 0.02, n).astype(F32)
    m = rng.normal(0, 1e-3, n).astype(F32)
    cm, am = q8.quantize_blockwise(m, maps.smap, maps.sthr)
    back = q8.dequantize(cm, am, maps.smap)
    rel = np.max(np.abs(back - m)) / np.max(np.abs(m))
    assert 1e-4 < rel < 2e-2


@pytest.mark.parametrize("bad", [math.inf, -math.inf, math.nan])
def test_q8_skip(maps, bad):
    rng = np.random.default_rng(11)
    n = 300
    p = rng.normal(0, 0.02, n).astype(F32)
    g = (rng.normal(0, 1e-3, n) * 65536).astype(F32)
    g[7] = bad
    cm = rng.integers(0, 256, n).astype(np.uint8)
    cv = rng.integers(0, 256, n).astype(np.uint8)
    am = np.ones(2, F32)
    av = np.ones(2, F32)
    before = [a.copy() for a in (p, cm, cv, am, av)]
    ok = q8.step_f32(p, g, cm, cv, am, av, lr=0.1, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1,
                     t=3, grad_scale=65536.0, maps=maps)
    assert ok is False
    for a, b in zip((p, cm, cv, am, av), before):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e30, 3e-20, 1e-30, 1e-39])
def test_normalise_is_ratio_within_one_ulp(scale):
    """x * fl(1/A) (with the 2**64 pre-scaling below 2**-64) stays within about
    one ulp of the exact ratio x / A, also for tiny and subnormal absmax."""
    rng = np.random.default_rng(17)
    xb = (rng.uniform(-1, 1, 256) * scale).astype(F32)
    a = q8.absmax_bits(xb)
    got = q8.normalise(xb, a).astype(np.float64)
    exact = xb.astype(np.float64) / np.float64(a)
    assert np.all(np.abs(got) <= 1.0)
    assert np.all(np.abs(got - exact) <= 2.5 * 2.0 ** -24 * np.maximum(np.abs(exact), 2.0 ** -126))
    # the element holding the absmax maps to exactly +-1 whenever 1/A is exact
    if a == F32(2.0) ** int(np.log2(a)):
        assert np.max(np.abs(got)) == 1.0
