"""Pins for the 4-bit code maps, nibble packing and the 4-bit-state step (CPU only).

The map contents are *parity unpinned* by the pages (they name torchao's
AdamW4bit, "4 bit Adam should support non constant lr", without its format);
pinned are the structure of the reading taken (the dynamic tree at 4 bits for
m: 7 magnitudes per sign in decades 1, 0.1, 0.01 holding 4, 2, 1 values;
k/16 without zero for v), the threshold quantiser against brute force, the
packing order, and the step against the first-step closed form of "Fix
decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
(bitsandbytes PR #2040) -- the update uses the dequantised state, and a zero
state (absmax 0) dequantises to exactly 0 whatever its codes.
"""

import math

import numpy as np
import pytest

from oracle import adamw as A
from oracle import q4, q8, qmap

F32 = np.float32


@pytest.fixture(scope="module")
def maps():
    return q4.Maps4()


def test_signed_map_structure(maps):
    t = maps.smap
    assert t.dtype == F32 and t.size == 16 and np.all(np.diff(t) > 0)
    assert t[-1] == 1.0 and 0.0 in t and t[0] > -1.0
    pos = t[(t > 0) & (t < 1)]
    assert np.array_equal(pos, -t[(t < 0)][::-1])        # symmetric apart from +1.0
    # decade counts of the dynamic tree at 3 magnitude bits: 1, 2, 4 values
    for lo, hi, count in ((0.001, 0.01, 1), (0.01, 0.1, 2), (0.1, 1.0, 4)):
        assert np.sum((pos >= lo) & (pos < hi)) == count
    # in each decade the values are the centres of equal bins of [0.1, 1] * decade
    assert pos[0] == F32(0.55 * 0.01)
    assert np.allclose(pos[1:3], [0.0325, 0.0775], rtol=2.0 ** -24, atol=0)
    assert np.allclose(pos[3:], [0.2125, 0.4375, 0.6625, 0.8875], rtol=2.0 ** -24, atol=0)


def test_unsigned_map_is_linear_without_zero(maps):
    t = maps.umap
    assert t.size == 16 and 0.0 not in t
    assert np.array_equal(t.astype(np.float64) * 16, np.arange(1, 17))


def _probe_points(table, thr, rng):
    pts = [table, thr, np.nextafter(thr, F32(-np.inf)),
           rng.uniform(-1.2, 1.2, 4000).astype(F32),
           (rng.standard_normal(2000) * 10.0 ** rng.uniform(-8, 0, 2000)).astype(F32),
           np.array([0.0, -0.0, 1.0, -1.0, 2.0, -2.0, 1e-30, -1e-30], F32)]
    return np.concatenate([np.asarray(p, F32) for p in pts])


@pytest.mark.parametrize("which", ["smap", "umap"])
def test_threshold_quantiser_equals_bruteforce(maps, which):
    table = getattr(maps, which)
    thr = qmap.thresholds(table)
    assert thr.size == 15
    x = _probe_points(table, thr, np.random.default_rng(21))
    assert np.array_equal(qmap.quantize(x, table, thr), qmap.quantize_bruteforce(x, table))


def test_map_values_quantise_to_themselves(maps):
    for table in (maps.smap, maps.umap):
        assert np.array_equal(qmap.quantize(table, table), np.arange(16))


def test_pack_order_and_roundtrip():
    assert np.array_equal(q4.pack(np.array([1, 2, 3], np.uint8)), np.array([0x21, 0x03], np.uint8))
    rng = np.random.default_rng(22)
    for n in (1, 2, 127, 128, 129, 1001):
        c = rng.integers(0, 16, n).astype(np.uint8)
        p = q4.pack(c)
        assert p.size == (n + 1) // 2
        assert np.array_equal(q4.unpack(p, n), c)
    with pytest.raises(ValueError):
        q4.pack(np.array([16], np.uint8))


def test_blockwise_roundtrip_error_bound(maps):
    rng = np.random.default_rng(23)
    x = (rng.normal(0, 1e-3, 1000) * rng.uniform(0, 1, 1000)).astype(F32)
    for table, thr, xx in ((maps.smap, maps.sthr, x), (maps.umap, maps.uthr, np.abs(x))):
        codes, amax = q4.quantize_blockwise(xx, table, thr)
        assert amax.size == 8  # 7 x 128 + 104
        y = q8.dequantize(codes, amax, table, q4.BLOCK)
        t = table.astype(np.float64)
        # nearest code: at most half the gap to a neighbour, or the distance
        # from the end codes to the ends of the range they cover
        gap = np.maximum(np.diff(t, prepend=t[0])[codes], np.diff(t, append=t[-1])[codes])
        edge = np.where(codes == 0, t[0] - (-1.0 if t[0] < 0 else 0.0), 0.0)
        bound = np.maximum(0.5 * gap, edge)
        a = amax[np.arange(xx.size) // q4.BLOCK].astype(np.float64)
        assert np.all(np.abs(y - xx) <= bound * a * (1 + 1e-5) + 1e-12)


def test_zero_blocks(maps):
    x = np.zeros(300, F32)
    cm, am = q4.quantize_blockwise(x, maps.smap, maps.sthr)
    assert np.all(am == 0) and np.all(cm == qmap.zero_code(maps.smap))
    cv, av = q4.quantize_blockwise(x, maps.umap, maps.uthr)
    assert np.all(av == 0) and np.all(cv == 0)   # no zero in the v map: code 0, absmax 0
    assert np.all(q8.dequantize(cv, av, maps.umap, q4.BLOCK) == 0)


def test_small_v_does_not_quantise_to_zero(maps):
    """The point of the zero-free v map: a tiny v in a block keeps 1/16 of the absmax."""
    v = np.full(128, 1e-12, F32)
    v[0] = 1.0
    cv, av = q4.quantize_blockwise(v, maps.umap, maps.uthr)
    back = q8.dequantize(cv, av, maps.umap, q4.BLOCK)
    assert np.all(back[1:] == F32(1 / 16)) and back[0] == 1.0


def _closed_form(p, g, lr, wd, eps):
    return p * (1 - lr * wd) - lr * g / (np.abs(g) + eps)


def test_first_step_closed_form_q4(maps):
    rng = np.random.default_rng(24)
    n = 1001
    p = rng.normal(0, 0.02, n).astype(F32)
    g = rng.normal(0, 1e-3, n).astype(F32)
    hp = dict(lr=A.f32(0.1), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8),
              wd=A.f32(0.1), t=1)
    nb = q8.n_blocks(n, q4.BLOCK)
    pm = rng.integers(0, 256, (n + 1) // 2).astype(np.uint8)   # any codes: absmax 0
    pv = rng.integers(0, 256, (n + 1) // 2).astype(np.uint8)
    am, av = np.zeros(nb, F32), np.zeros(nb, F32)
    p32 = p.copy()
    assert q4.step_f32(p32, g, pm, pv, am, av, maps=maps, **hp)
    want = _closed_form(p.astype(np.float64), g.astype(np.float64), hp["lr"], hp["wd"], hp["eps"])
    assert np.max(np.abs(p32 - want) / (np.abs(want) + hp["lr"])) < 8 * 2.0 ** -24
    p64, _, _ = q4.step_fp64(p, g, (np.zeros_like(pm), np.zeros(nb, F32)),
                             (np.zeros_like(pv), np.zeros(nb, F32)), maps=maps, **hp)
    assert np.allclose(p64, want, rtol=1e-13, atol=1e-16)
    assert np.array_equal(am, np.array([q8.absmax_bits(F32(1 - F32(0.9)) * g[i * 128:(i + 1) * 128])
                                        for i in range(nb)], F32))
    assert pm[-1] >> 4 == 0 and pv[-1] >> 4 == 0          # odd n: last high nibble 0


def test_q4_update_uses_unquantised_moments(maps):
    rng = np.random.default_rng(25)
    n = 256
    p = rng.normal(0, 0.02, n).astype(F32)
    g = rng.normal(0, 1e-3, n).astype(F32)
    cm = rng.integers(0, 16, n).astype(np.uint8)
    cv = rng.integers(0, 16, n).astype(np.uint8)
    am = np.array([1e-3, 2e-3], F32)
    av = np.array([1e-6, 3e-6], F32)
    m = q8.dequantize(cm, am, maps.smap, q4.BLOCK)
    v = q8.dequantize(cv, av, maps.umap, q4.BLOCK)
    hp = dict(lr=A.f32(1e-3), beta1=A.f32(0.9), beta2=A.f32(0.999), eps=A.f32(1e-8))
    x = A.Tensor(p=p.copy(), g=g, m=m.copy(), v=v.copy(), wd=A.f32(0.01))
    A.step_f32([x], t=4, **hp)
    p4 = p.copy()
    pm, pv = q4.pack(cm), q4.pack(cv)
    q4.step_f32(p4, g, pm, pv, am, av, wd=A.f32(0.01), t=4, maps=maps, **hp)
    assert np.array_equal(p4, x.p)
    assert np.array_equal(q4.unpack(pm, n), q4.quantize_blockwise(x.m, maps.smap, maps.sthr)[0])
    assert np.array_equal(q4.unpack(pv, n), q4.quantize_blockwise(x.v, maps.umap, maps.uthr)[0])


def test_block_independence(maps):
    rng = np.random.default_rng(26)
    x = rng.normal(0, 1e-3, 512).astype(F32)
    c0, a0 = q4.quantize_blockwise(x, maps.smap, maps.sthr)
    y = x.copy()
    y[130] *= 50                                         # inside the second block only
    c1, a1 = q4.quantize_blockwise(y, maps.smap, maps.sthr)
    same = np.r_[0:128, 256:512]
    assert np.array_equal(c0[same], c1[same]) and a0[0] == a1[0] and np.array_equal(a0[2:], a1[2:])
    assert a1[1] != a0[1]


@pytest.mark.parametrize("bad", [math.inf, -math.inf, math.nan])
def test_q4_skip(maps, bad):
    rng = np.random.default_rng(27)
    n = 300
    p = rng.normal(0, 0.02, n).astype(F32)
    g = (rng.normal(0, 1e-3, n) * 65536).astype(F32)
    g[7] = bad
    pm = rng.integers(0, 256, 150).astype(np.uint8)
    pv = rng.integers(0, 256, 150).astype(np.uint8)
    am, av = np.ones(3, F32), np.ones(3, F32)
    before = [a.copy() for a in (p, pm, pv, am, av)]
    assert q4.step_f32(p, g, pm, pv, am, av, lr=0.1, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1,
                       t=3, grad_scale=65536.0, maps=maps) is False
    for a, b in zip((p, pm, pv, am, av), before):
        assert np.array_equal(a, b)
