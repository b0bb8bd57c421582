"""The two float32 readings this library takes for speed, against the plain forms.

The workload writes the 8-bit re-quantisation as the nearest code of
x = m'/A, and the AdamWMini listing of "Adam-mini <> DTensor" writes the
bias-corrected denominator as sqrt(v')/sqrt(bc2) + eps.  The library (and the
strict-fp32 oracle that mirrors it bit for bit) instead forms
x = m' * fl(1/A) with one reciprocal per block, and h = sqrt(v') *
fl(1/sqrt(bc2)) + eps with one reciprocal per launch: fewer instructions in
kernels that are bound by instruction issue.  These tests bound what that
choice can change, against the plain division forms the oracle also holds:

  * a code moves by exactly one, and only where the exact ratio m'/A lies
    within 2.5 ulp of a threshold between two codes (the reciprocal form is
    within 1.5 ulp of the exact ratio, the division within 0.5 ulp) --
    checked on every float32 within 4 ulp of every threshold of the default
    8-bit and 4-bit maps, for many block maxima, and on random blocks;
  * on the states of twenty 8-bit steps the same holds, at a rate of about
    one code in 10^5 or fewer;
  * one step from the same state moves the parameter by the division form's
    result within 2 ulp plus 8 x 2^-24 of the step term, and both forms stay
    within the float64 definition's 5e-5 after ten steps at lr = wd = 0.1.

The measured rates of differing codes are printed (run with -s).
"""

import os

import numpy as np
import pytest

from oracle import adamw as OA
from oracle import q8, qmap as qm

F32 = np.float32
EXHAUSTIVE = os.environ.get("ADAMW_EXHAUSTIVE") == "1"


def _ulp(x):
    x = np.abs(np.asarray(x, F32))
    return (np.nextafter(x, F32(np.inf)) - x).astype(np.float64)


def _compare(mb, a, table, thr):
    """Codes of the values mb (one block maximum a) under both rules; checks the bound and
    returns (values compared, codes that differ)."""
    x_div = q8.normalise(mb, a, "division")
    x_mul = q8.normalise(mb, a, "reciprocal")
    c_div = qm.quantize(x_div, table, thr).astype(np.int64)
    c_mul = qm.quantize(x_mul, table, thr).astype(np.int64)
    diff = np.nonzero(c_div != c_mul)[0]
    if diff.size:
        assert np.all(np.abs(c_div[diff] - c_mul[diff]) == 1)
        t = thr[np.minimum(c_div[diff], c_mul[diff])].astype(np.float64)
        exact = mb[diff].astype(np.float64) / np.float64(a)
        assert np.all(np.abs(exact - t) <= 2.5 * _ulp(t)), "a code moved away from any threshold"
    return mb.size, diff.size


def _maps():
    out = [("signed 8-bit", qm.signed_map()), ("unsigned 8-bit", qm.unsigned_map()),
           ("signed 4-bit", qm.signed_map4()), ("unsigned 4-bit", qm.unsigned_map4())]
    return [(name, t, qm.thresholds(t)) for name, t in out]


@pytest.mark.parametrize("name,table,thr", _maps(), ids=lambda x: x if isinstance(x, str) else "")
def test_codes_near_every_threshold(name, table, thr):
    """Every float32 within 4 ulp of each threshold, as the ratio of m' = fl(x * A) and A
    for 64 block maxima A spread over 60 binades."""
    rng = np.random.default_rng(31)
    a_vals = (2.0 ** rng.uniform(-60, 0, 64) * rng.uniform(1, 2, 64)).astype(F32)
    n_all = n_diff = 0
    for t in thr:
        xs = [t]
        lo = hi = t
        for _ in range(4):
            lo = np.nextafter(lo, F32(-np.inf))
            hi = np.nextafter(hi, F32(np.inf))
            xs += [lo, hi]
        xs = np.array(xs, F32)
        xs = xs[np.abs(xs) <= 1]
        for a in a_vals:
            mb = (xs * a).astype(F32)
            mb = mb[np.abs(mb) <= a]
            n, d = _compare(mb, a, table, thr)
            n_all += n
            n_diff += d
    print(f"{name}: {n_diff} of {n_all} codes within 4 ulp of a threshold differ")
    assert n_diff < n_all


@pytest.mark.parametrize("name,table,thr", _maps()[:2], ids=lambda x: x if isinstance(x, str) else "")
def test_codes_of_random_blocks(name, table, thr):
    """Random 256-element blocks with the magnitudes an optimizer state takes
    (log-uniform block scales over 40 decades): 4e4 blocks, 1e7 with ADAMW_EXHAUSTIVE=1."""
    rng = np.random.default_rng(32)
    n_blocks = 10 ** 7 if EXHAUSTIVE else 40_000
    n_all = n_diff = 0
    per = 20_000
    for start in range(0, n_blocks, per):
        k = min(per, n_blocks - start)
        scale = 10.0 ** rng.uniform(-40, 0, (k, 1))
        x = rng.standard_normal((k, 256)) * scale
        if "unsigned" in name:
            x = x * x
        x = x.astype(F32)
        amax = (x.view(np.uint32) & np.uint32(0x7FFFFFFF)).max(axis=1).view(F32)
        keep = amax > 0
        x, amax = x[keep], amax[keep]
        # division form per row; reciprocal form per row (scaled rows where A < 2**-64)
        x_div = (x / amax[:, None]).astype(F32)
        small = amax < q8.SMALL
        s = np.where(small, q8.SCALE, F32(1.0)).astype(F32)
        y = (F32(1.0) / (amax * s).astype(F32)).astype(F32)
        x_mul = ((x * s[:, None]).astype(F32) * y[:, None]).astype(F32)
        c_div = qm.quantize(x_div.ravel(), table, thr).astype(np.int64)
        c_mul = qm.quantize(x_mul.ravel(), table, thr).astype(np.int64)
        diff = np.nonzero(c_div != c_mul)[0]
        if diff.size:
            assert np.all(np.abs(c_div[diff] - c_mul[diff]) == 1)
            t = thr[np.minimum(c_div[diff], c_mul[diff])].astype(np.float64)
            exact = x.ravel()[diff].astype(np.float64) / np.repeat(amax, 256)[diff].astype(np.float64)
            assert np.all(np.abs(exact - t) <= 2.5 * _ulp(t))
        n_all += c_div.size
        n_diff += diff.size
    print(f"{name}: {n_diff} of {n_all} codes of random blocks differ ({n_diff / n_all:.2e})")
    assert n_diff <= 1e-4 * n_all


def test_8bit_steps_under_both_rules():
    """Twenty 8-bit steps from zero state, bf16-sized grads: at every step the
    re-quantisation of the same m', v' under both rules.  Codes differ in a
    small fraction of elements, by one, each next to a threshold."""
    rng = np.random.default_rng(33)
    n = 256 * 512
    maps = q8.Maps()
    p = rng.normal(0, 0.02, n).astype(F32)
    cm, cv = np.zeros(n, np.uint8), np.zeros(n, np.uint8)
    am, av = np.zeros(n // 256, F32), np.zeros(n // 256, F32)
    n_diff = [0, 0]
    for t in range(1, 21):
        g = rng.normal(0, 1e-3, n).astype(F32)
        s = OA.f32_scalars(lr=OA.f32(1e-3), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                           eps=OA.f32(1e-8), t=t)
        m = q8.dequantize(cm, am, maps.smap)
        v = q8.dequantize(cv, av, maps.umap)
        _, m1, v1 = OA.elementwise_f32(p, g, m, v, s, OA.decay_f32(s.lr, OA.f32(0.01)))
        for k, (x, table, thr) in enumerate(((m1, maps.smap, maps.sthr), (v1, maps.umap, maps.uthr))):
            for b in range(n // 256):
                xb = x[b * 256:(b + 1) * 256]
                a = q8.absmax_bits(xb)
                if a > 0:
                    n_diff[k] += _compare(xb, a, table, thr)[1]
        q8.step_f32(p, g, cm, cv, am, av, lr=OA.f32(1e-3), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                    eps=OA.f32(1e-8), wd=OA.f32(0.01), t=t, maps=maps)
    print(f"20 steps x {n} elements: {n_diff[0]} m codes and {n_diff[1]} v codes differ")
    assert sum(n_diff) <= 1e-4 * 2 * 20 * n


@pytest.mark.parametrize("lr,wd", [(0.1, 0.1), (1e-3, 0.01)])
def test_bias_correction_division_form(lr, wd):
    """h = sqrt(v')/sqrt(bc2) + eps against sqrt(v')*fl(1/sqrt(bc2)) + eps over 10 steps:
    from the same state the two forms give params within 2 ulp of p' plus 8 x 2^-24
    of the step term, and both trajectories stay within 5e-5 of the float64 definition
    after 10 steps."""
    rng = np.random.default_rng(35)
    n = 1 << 18
    p0 = rng.normal(0, 0.02, n).astype(F32)
    forms = {k: OA.Tensor(p=p0.copy(), g=None, m=np.zeros(n, F32), v=np.zeros(n, F32), wd=OA.f32(wd))
             for k in ("reciprocal", "division")}
    ref = OA.Tensor(p=p0.astype(np.float64), g=None, m=np.zeros(n), v=np.zeros(n), wd=OA.f32(wd))
    worst_ulps = 0.0
    for t in range(1, 11):
        g = rng.normal(0, 1e-3, n).astype(F32)
        ref.g = g.astype(np.float64)
        OA.step_fp64([ref], lr=OA.f32(lr), beta1=OA.f32(0.9), beta2=OA.f32(0.999), eps=OA.f32(1e-8), t=t)
        before = {k: (x.p.copy(), x.m.copy(), x.v.copy()) for k, x in forms.items()}
        for rule, x in forms.items():
            s = OA.f32_scalars(lr=OA.f32(lr), beta1=OA.f32(0.9), beta2=OA.f32(0.999),
                               eps=OA.f32(1e-8), t=t)
            x.p[...], x.m[...], x.v[...] = OA.elementwise_f32(x.p, g, x.m, x.v, s,
                                                              OA.decay_f32(s.lr, x.wd), bias_rule=rule)
        # one step from the same state: the two forms differ by a few ulp at most
        s = OA.f32_scalars(lr=OA.f32(lr), beta1=OA.f32(0.9), beta2=OA.f32(0.999), eps=OA.f32(1e-8), t=t)
        p_a, _, _ = OA.elementwise_f32(*before["reciprocal"][:1], g, *before["reciprocal"][1:], s,
                                       OA.decay_f32(s.lr, OA.f32(wd)), bias_rule="reciprocal")
        p_b, _, _ = OA.elementwise_f32(*before["reciprocal"][:1], g, *before["reciprocal"][1:], s,
                                       OA.decay_f32(s.lr, OA.f32(wd)), bias_rule="division")
        # |p_a - p_b| against the size of the step term lr*|u| (p_old*decay - p'), in
        # units of 2**-24: the denominators differ by about 2.5 ulp, the quotient and
        # the product each add one rounding, and the final subtraction one ulp of p'
        p_old = before["reciprocal"][0]
        term = np.abs((p_old * OA.decay_f32(s.lr, OA.f32(wd))).astype(np.float64) - p_a)
        excess = np.abs(p_a.astype(np.float64) - p_b.astype(np.float64)) - 2 * _ulp(p_a)
        ratio = np.max(np.maximum(excess, 0) / np.maximum(term, 1e-300)) / 2.0 ** -24
        worst_ulps = max(worst_ulps, float(ratio))
    assert worst_ulps <= 8
    for x in forms.values():
        assert np.max(np.abs(x.p.astype(np.float64) - ref.p)) <= 5e-5
    print(f"lr={lr} wd={wd}: single steps differ by at most {worst_ulps:.1f} x 2^-24 of the step term")
