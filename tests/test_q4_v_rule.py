"""The closed-form nearest-code rule for the 4-bit second moment (CPU only).

The 4-bit step does not search a table for v: its map is k/16 (code k-1),
whose thresholds are the exact midpoints (k + 1.5)/16, so for a normalised
float32 x the code is clamp(ceil(fl32(16x - 1.5)), 0, 15) -- one fused
multiply-add rounded once to float32, a round-up conversion, a clamp, NaN
to code 0.  This file checks that identity against the oracle's threshold
rule (``qmap.quantize``, itself pinned against brute-force nearest) on every
float32 within 2048 ulps of each threshold and of each map value, on a
million random floats of [0, 1], and on the special values; the sweep over
every float32 of [0, 1.01] runs with ADAMW_EXHAUSTIVE=1.  The fma is
emulated exactly: 16x is exact in float64, 16x - 1.5 is exact in float64 for
x >= 2^-33, and below that both roundings give -1.5 (code 0).
"""

import os

import numpy as np
import pytest

from oracle import q4, qmap

F32 = np.float32


def closed_form(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=F32)
    with np.errstate(invalid="ignore"):
        t = (x.astype(np.float64) * 16.0 - 1.5).astype(F32)     # the fma, one float32 rounding
        c = np.ceil(t.astype(np.float64))
        c = np.where(np.isnan(c), 0.0, c)                       # NaN converts to 0
    return np.clip(c, 0, 15).astype(np.uint8)


@pytest.fixture(scope="module")
def table():
    m = q4.Maps4()
    return m.umap, m.uthr


def _neighbours(v: np.ndarray, span: int) -> np.ndarray:
    bits = np.asarray(v, dtype=F32).view(np.int32).astype(np.int64)
    out = (bits[:, None] + np.arange(-span, span + 1)[None, :]).ravel()
    out = out[(out >= 0) & (out <= 0x3F810000)]                  # [0, 1.0078] as float bits
    return out.astype(np.int32).view(F32)


def test_closed_form_matches_thresholds_near_every_boundary(table):
    umap, uthr = table
    x = np.concatenate([_neighbours(uthr, 2048), _neighbours(umap, 2048)])
    assert np.array_equal(closed_form(x), qmap.quantize(x, umap, uthr))


def test_closed_form_matches_thresholds_on_random_floats(table):
    umap, uthr = table
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(0, 1, 1 << 20).astype(F32),
                        (rng.uniform(0, 1, 1 << 18) ** 8).astype(F32),     # small magnitudes
                        rng.integers(0, 0x3F800001, 1 << 18).astype(np.int32).view(F32)])
    assert np.array_equal(closed_form(x), qmap.quantize(x, umap, uthr))


def test_closed_form_special_values(table):
    umap, uthr = table
    x = np.array([0.0, -0.0, 1.0, np.nextafter(F32(1), F32(2)), 1e-45, 2.0 ** -126, 0.09375,
                  0.15625, 1.5 / 16, 2.5 / 16, 15.5 / 16, np.nan], dtype=F32)
    got = closed_form(x)
    assert np.array_equal(got, qmap.quantize(x, umap, uthr))
    assert got[0] == 0 and got[1] == 0 and got[2] == 15 and got[3] == 15 and got[-1] == 0
    assert got[8] == 0 and got[9] == 1 and got[10] == 14          # exact midpoints: the lower code


@pytest.mark.skipif(os.environ.get("ADAMW_EXHAUSTIVE") != "1",
                    reason="set ADAMW_EXHAUSTIVE=1 (every float32 of [0, 1.01], about a minute)")
def test_closed_form_matches_thresholds_on_every_float(table):
    umap, uthr = table
    step = 1 << 24
    for lo in range(0, 0x3F810001, step):
        x = np.arange(lo, min(lo + step, 0x3F810001), dtype=np.int64).astype(np.int32).view(F32)
        assert np.array_equal(closed_form(x), qmap.quantize(x, umap, uthr)), hex(lo)
