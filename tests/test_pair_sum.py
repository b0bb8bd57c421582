"""The accuracy of the Adam-mini block reduction's summation method (CPU only).

The GPU reduction sums g*g over a block without a float64 operation per
element: every lane sums the 32 squares of one round of its loads as an
unevaluated pair of float32 (s, c) -- each square split exactly into
x*x = p + e (one fma), each addition into s made error-free by TwoSum, the
errors gathered in c (Ogita, Rump and Oishi, "Accurate sum and dot product",
2005) -- and the pairs are added in float64.  This file emulates that method
in numpy float32 arithmetic (every operation rounded once, as on the GPU; the
fma's error term is exact in float64) over chains of 32 squares, and checks it
against the exactly rounded sum (``math.fsum``): the relative
error stays below 2^-40 on wide-range and on cancellation-free data alike,
far inside the one float32 ulp (2^-24) at which the block mean is stored.
A plain float32 running sum, for contrast, is off by about 2^-20 already.
"""

import math

import numpy as np

F32 = np.float32


def two_product_square(x):
    p = (x * x).astype(F32)
    e = (x.astype(np.float64) * x.astype(np.float64) - p.astype(np.float64)).astype(F32)  # exact
    return p, e


def two_sum(a, b):
    t = (a + b).astype(F32)
    bp = (t - a).astype(F32)
    err = ((a - (t - bp).astype(F32)).astype(F32) + (b - bp).astype(F32)).astype(F32)
    return t, err


def pair_sum(x: np.ndarray, chain: int = 32) -> float:
    """Sum of x*x: chains of `chain` squares in float32 pairs, chains added in float64."""
    x = np.asarray(x, dtype=F32).reshape(-1, chain)
    s = np.zeros(x.shape[0], F32)
    c = np.zeros(x.shape[0], F32)
    for j in range(chain):
        p, e = two_product_square(x[:, j])
        s, err = two_sum(s, p)
        c = (c + (err + e).astype(F32)).astype(F32)
    return float(np.sum(s.astype(np.float64)) + np.sum(c.astype(np.float64)))


def exact_sum_of_squares(x: np.ndarray) -> float:
    xd = np.asarray(x, dtype=F32).astype(np.float64)
    return math.fsum(xd * xd)          # every square exact in float64, the sum correctly rounded


def test_pair_sum_is_accurate_on_a_head_sized_block():
    rng = np.random.default_rng(7)
    x = (rng.normal(0, 1e-3, 524_288) * rng.uniform(0.1, 10, 524_288)).astype(F32)
    ref = exact_sum_of_squares(x)
    assert abs(pair_sum(x) - ref) / ref < 2.0 ** -40
    naive = np.float32(0)
    for v in (x * x).astype(F32)[:65536]:
        naive = np.float32(naive + v)
    part = exact_sum_of_squares(x[:65536])
    assert abs(float(naive) - part) / part > 2.0 ** -22   # what the pairs avoid


def test_pair_sum_is_accurate_on_wide_ranges():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(1 << 18) * np.exp2(rng.uniform(-40, 10, 1 << 18))).astype(F32)
    ref = exact_sum_of_squares(x)
    assert abs(pair_sum(x) - ref) / ref < 2.0 ** -40


def test_pair_sum_of_equal_values():
    x = np.full(16384, F32(3e-3))       # a float32 running sum drifts most on equal terms
    ref = exact_sum_of_squares(x)
    assert abs(pair_sum(x) - ref) / ref < 2.0 ** -40


def test_unscaled_16bit_squares_are_exact_in_float32():
    """The reduction skips the product's error term for unscaled bf16 and fp16
    grads: every one of their 65,536 patterns squares exactly in float32
    wherever the square is a normal float32 (8 or 11 significant bits squared
    fit in 24); a square below that range or past it is where the header's
    bound and the float64 fallback take over."""
    bf = (np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)).view(np.float32)
    hf = np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(F32)
    tiny, big = np.finfo(F32).tiny, np.finfo(F32).max
    for x in (bf, hf):
        x = x[np.isfinite(x)]
        exact = x.astype(np.float64) ** 2
        normal = (exact >= tiny) & (exact <= big)
        with np.errstate(over="ignore", under="ignore"):
            sq = (x * x).astype(F32)
        assert np.array_equal(sq[normal].astype(np.float64), exact[normal])
        assert normal.sum() > 20000
