"""Pins for the remainder split/join oracle (CPU only).

"Support store_param_remainders feature from Apex in TE Fused Adam #1408",
Description: the fp32 master is rebuilt from the bf16 model param plus its 16
trailing remainder bits.  Pinned here by brute force (every top half against
a boundary set of low halves, and every low half against a boundary set of top
halves; the full 2**32 sweep runs with ADAMW_EXHAUSTIVE=1), by an independent
nearest-ties-away rounding computed from exact distances, and by torch's own
round-to-nearest-even conversion, which must agree everywhere but at ties.
"""

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import remainder as R

LO_SET = np.array([0x0000, 0x0001, 0x3FFF, 0x4000, 0x7FFE, 0x7FFF, 0x8000, 0x8001,
                   0xBFFF, 0xC000, 0xFFFE, 0xFFFF], dtype=np.uint32)


def _grid(tops, los):
    tops = np.asarray(tops, np.uint32)[:, None]
    los = np.asarray(los, np.uint32)[None, :]
    return ((tops << np.uint32(16)) | los).ravel()


def _roundtrip_ok(bits):
    """join(split(x)) is x for every master but a NaN; a NaN master is stored as
    the quiet NaN (bf16 half 0x7FC0, a NaN; remainder 0) and comes back as it."""
    hi, rem = R.split(bits)
    back = R.join(hi, rem).view(np.uint32)
    nan = (bits & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    return (np.array_equal(back[~nan], bits[~nan]) and np.all(back[nan] == 0x7FC00000)
            and np.all(hi[nan] == 0x7FC0) and np.all(rem[nan] == 0))


def test_roundtrip_all_top_halves():
    rng = np.random.default_rng(0)
    los = np.concatenate([LO_SET, rng.integers(0, 1 << 16, 52, dtype=np.uint32)])
    assert _roundtrip_ok(_grid(np.arange(1 << 16), los))


def test_roundtrip_all_low_halves():
    tops = [0x0000, 0x0001, 0x007F, 0x0080, 0x3F80, 0x7F7F, 0x7F80, 0x7FC0, 0x7FFF,
            0x8000, 0x8001, 0xBF80, 0xFF7F, 0xFF80, 0xFFFF]
    assert _roundtrip_ok(_grid(tops, np.arange(1 << 16)))


@pytest.mark.skipif(os.environ.get("ADAMW_EXHAUSTIVE") != "1", reason="set ADAMW_EXHAUSTIVE=1 (about 2 min)")
def test_roundtrip_exhaustive():
    n = 1 << 24
    base = np.arange(n, dtype=np.uint32)
    for c in range(256):
        assert _roundtrip_ok(base + np.uint32(c * n))


def _nearest_ties_away(x: float) -> int:
    """bf16 bits nearest to finite x, ties away from zero, from exact distances."""
    b = int(np.float32(x).view(np.uint32))
    sign, mag = b & 0x80000000, b & 0x7FFFFFFF
    down = mag & 0xFFFF0000                    # truncated magnitude
    up = down + 0x10000                        # next bf16 magnitude (0x7F800000 = inf)
    fx = abs(Fraction(float(np.uint32(mag).view(np.float32))))
    fd = Fraction(float(np.uint32(down).view(np.float32)))
    # the value "one bf16 step above the largest finite" is 2**128 for rounding purposes
    fu = Fraction(2) ** 128 if up == 0x7F800000 else Fraction(float(np.uint32(up).view(np.float32)))
    pick = up if (fx - fd) >= (fu - fx) else down
    return (sign | pick) >> 16


def test_bf16_half_is_nearest_ties_away():
    rng = np.random.default_rng(1)
    bits = np.concatenate([
        rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32),
        _grid([0x0000, 0x0001, 0x3F80, 0x3F81, 0x7F7F, 0x8001, 0xBF80, 0xFF7F], LO_SET),
    ])
    x = bits.view(np.float32)
    finite = np.isfinite(x)
    hi, _ = R.split(bits)
    for b, h in zip(bits[finite], hi[finite]):
        assert int(h) == _nearest_ties_away(float(np.uint32(b).view(np.float32))), hex(int(b))


def test_bf16_half_agrees_with_torch_except_ties():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, 1 << 20).astype(np.float32)
    x[:1000] = rng.normal(0, 1e-38, 1000).astype(np.float32)  # subnormals
    hi, _ = R.split(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    tie = (x.view(np.uint32) & 0xFFFF) == 0x8000
    assert np.array_equal(hi[~tie], ref[~tie])
    # at an exact tie: ours rounds away from zero, torch to even -- they differ only there
    assert np.all(np.abs(hi[tie].astype(np.int32) - ref[tie].astype(np.int32)) <= 1)


def test_special_values_round_trip_and_bf16_view():
    vals = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -1.0,
                     np.finfo(np.float32).tiny, np.finfo(np.float32).max,
                     np.float32(1e-45), -np.float32(1e-45)], dtype=np.float32)
    hi, rem = R.split(vals)
    back = R.join(hi, rem)
    assert np.array_equal(back.view(np.uint32), vals.view(np.uint32))
    bf = R.bf16_bits_to_f32(hi)
    # zeros stay (signed) zeros with a zero remainder; infinities stay infinities
    assert bf[0] == 0 and not np.signbit(bf[0]) and rem[0] == 0
    assert bf[1] == 0 and np.signbit(bf[1]) and rem[1] == 0
    assert bf[2] == np.inf and bf[3] == -np.inf and np.isnan(bf[4])
    assert bf[5] == 1.0 and bf[6] == -1.0
    # FLT_MAX is past the last bf16 tie: rounds to inf, the remainder still rebuilds it
    assert bf[8] == np.inf and back[8] == np.finfo(np.float32).max


def test_every_nan_master_is_a_nan_in_the_bf16_half():
    """The all-ones NaNs -- 0x7FFFFFFF is the NaN a GPU's arithmetic returns --
    would carry out of the 16-bit half under the plain increment and read as
    -0.0 / +0.0; every NaN master must give a NaN bf16 model parameter."""
    tops = np.array([0x7F80, 0x7F81, 0x7FBF, 0x7FC0, 0x7FFE, 0x7FFF,
                     0xFF80, 0xFF81, 0xFFC0, 0xFFFE, 0xFFFF], dtype=np.uint32)
    bits = _grid(tops, np.arange(1 << 16, dtype=np.uint32))
    bits = bits[(bits & 0x7FFFFFFF) > 0x7F800000]          # NaNs only (drops the infinities)
    hi, rem = R.split(bits)
    assert np.all(np.isnan(R.bf16_bits_to_f32(hi)))
    assert np.all(hi == 0x7FC0) and np.all(rem == 0)
    assert np.all(R.join(hi, rem).view(np.uint32) == 0x7FC00000)
    gpu_nan = np.array([0x7FFFFFFF], dtype=np.uint32)
    assert np.isnan(R.bf16_bits_to_f32(R.split(gpu_nan)[0]))[0]


def test_remainder_sign_says_rounded_up():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 0.02, 4096).astype(np.float32)
    hi, rem = R.split(x)
    trunc = (x.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(hi != trunc, rem < 0)
