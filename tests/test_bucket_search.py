"""The bucketed nearest-code search of the 8-bit and 4-bit steps (CPU only).

The kernels do not binary-search the 255 thresholds of a map.  They split
|x| into buckets -- one for |x| < 2^-24, then 128 per binade from 2^-24 up to
2, keyed by the exponent and the top 7 mantissa bits, and a last one for
everything above (only NaN reaches it) -- and keep per bucket and sign the
lowest code any x of the bucket can have.  With at most R thresholds inside
any bucket, code = lo + #{r < R : thr[lo + r] <= x}.  This file rebuilds the
bucket tables from that definition (independently of the library's builder)
and checks the identity against the oracle's threshold rule
(``qmap.quantize``) for the default 8-bit maps and the 4-bit m map: near every
threshold, on random floats of [-1, 1], and, with ADAMW_EXHAUSTIVE=1, on
every float32 of [-1.01, 1.01].  It also checks that the default maps need a
single compare per lookup (R = 1), the case the kernels are tuned for.
"""

import os

import numpy as np
import pytest

from oracle import qmap

F32 = np.float32
N_BUCKETS = 1 + 25 * 128          # |x| < 2^-24, then 25 binades x 128
BASE = 103 * 128 - 1              # (exponent 103 = 2^-24, mantissa top 0) is bucket 1


def bucket(x: np.ndarray) -> np.ndarray:
    mag = np.asarray(x, dtype=F32).view(np.uint32) & np.uint32(0x7FFFFFFF)
    return np.clip((mag >> np.uint32(16)).astype(np.int64) - BASE, 0, N_BUCKETS - 1)


def bucket_bounds(k: int) -> tuple[float, float]:
    """Smallest and largest |x| of bucket k (the last bucket: from 2.0 up)."""
    if k == 0:
        return 0.0, float(np.uint32((103 << 23) - 1).view(F32))
    bits = (k + BASE) << 16
    return (float(np.uint32(bits).view(F32)), float(np.uint32(bits | 0xFFFF).view(F32)))


def tables(thr: np.ndarray):
    """lo_pos[k] / lo_neg[k]: the lowest code of any x >= 0 / x <= 0 in bucket k,
    and R, the most thresholds inside one bucket of either sign."""
    def count(x):
        return int(np.searchsorted(thr, F32(x), side="right"))
    lo_pos = np.zeros(N_BUCKETS, np.int64)
    lo_neg = np.zeros(N_BUCKETS, np.int64)
    r = 0
    for k in range(N_BUCKETS - 1):
        a, b = bucket_bounds(k)
        lo_pos[k], lo_neg[k] = count(a), count(-b)
        r = max(r, count(b) - count(a), count(-a) - count(-b))
    return lo_pos, lo_neg, max(r, 1)            # the last bucket (NaN) keeps code 0


def bucket_search(x, thr, lo_pos, lo_neg, r):
    x = np.asarray(x, dtype=F32)
    k = bucket(x)
    neg = np.signbit(x)
    lo = np.where(neg, lo_neg[k], lo_pos[k])
    pad = np.concatenate([thr, np.full(r + 1, np.inf, F32)])
    code = lo.copy()
    for i in range(r):
        code += (pad[lo + i] <= x)                 # NaN compares false
    return code.astype(np.uint8)


MAPS = {"8-bit m": qmap.signed_map, "8-bit v": qmap.unsigned_map, "4-bit m": qmap.signed_map4}


@pytest.fixture(scope="module", params=sorted(MAPS))
def setup(request):
    table = MAPS[request.param]()
    thr = qmap.thresholds(table)
    lo_pos, lo_neg, r = tables(thr)
    return request.param, table, thr, lo_pos, lo_neg, r


def test_default_maps_need_one_compare(setup):
    name, table, thr, lo_pos, lo_neg, r = setup
    assert r == 1, name


def _around(values, span):
    bits = np.asarray(values, dtype=F32).view(np.int32).astype(np.int64)
    out = (bits[:, None] + np.arange(-span, span + 1)[None, :]).ravel()
    return out.astype(np.int32).view(F32)


def test_search_matches_thresholds(setup):
    name, table, thr, lo_pos, lo_neg, r = setup
    rng = np.random.default_rng(1)
    x = np.concatenate([
        _around(thr, 256), _around(table, 256),
        rng.uniform(-1, 1, 1 << 20).astype(F32),
        (rng.uniform(-1, 1, 1 << 18) ** 9).astype(F32),
        np.array([0.0, -0.0, 1.0, -1.0, 2.0 ** -24, -(2.0 ** -24), 1e-45, np.nan, -np.nan], F32)])
    x = x[np.isnan(x) | (np.abs(x) <= 1.0078125)]
    want = qmap.quantize(x, table, thr)
    assert np.array_equal(bucket_search(x, thr, lo_pos, lo_neg, r), want), name


@pytest.mark.skipif(os.environ.get("ADAMW_EXHAUSTIVE") != "1",
                    reason="set ADAMW_EXHAUSTIVE=1 (every float32 of [-1.01, 1.01], about 5 minutes)")
def test_search_matches_thresholds_on_every_float(setup):
    name, table, thr, lo_pos, lo_neg, r = setup
    step = 1 << 24
    for sign in (0, 1 << 31):
        for lo in range(0, 0x3F810001, step):
            bits = np.arange(lo, min(lo + step, 0x3F810001), dtype=np.int64) | sign
            x = bits.astype(np.uint32).view(F32)
            assert np.array_equal(bucket_search(x, thr, lo_pos, lo_neg, r),
                                  qmap.quantize(x, table, thr)), (name, sign, hex(lo))
