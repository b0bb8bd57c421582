"""The GPU parity checks reject a step with the decay applied after the update.

"Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels"
(bitsandbytes PR #2040) fixed kernels that computed p = (p - lr*u)(1 - lr*wd)
instead of p*(1 - lr*wd) - lr*u, and checked its tests by re-registering the
wrong ordering and watching them fail.  Here the wrong ordering is planted in
the oracle, on the CPU (no kernel is built broken on purpose): its outputs are
handed, in place of the library's, to the acceptance checks that the GPU test
of the single-tensor workload applies (``tests/test_gpu_fp32.py``: bit-exact
against the strict-fp32 oracle every step, 1e-6 relative to the float64
definition on the first step, 5e-5 after ten steps at lr = wd = 0.1).  All
three reject it -- the first-step gap is lr * wd * lr * |u|, about 1.0e-3 --
and at wd = 0, where both orderings are the same arithmetic, all three pass.
"""

import numpy as np
import pytest

from oracle import adamw as OA
from _support import assert_max_abs, assert_single_step_rel, assert_state_bitexact

f32 = OA.f32
B1, B2, EPS = f32(0.9), f32(0.999), f32(1e-8)
N = 1 << 20   # the workload's single tensor


def _run(wd, decay_after, steps=10, lr=0.1):
    """Ten steps of the single-tensor workload: the strict-fp32 step (correct, or
    with the decay planted after the update), the correct strict-fp32 oracle and the
    float64 definition, on the same seeded inputs; the checks see each step."""
    rng = np.random.default_rng(1)
    p0 = rng.normal(0, 0.02, N).astype(np.float32)
    got = OA.Tensor(p=p0.copy(), g=None, m=np.zeros(N, np.float32), v=np.zeros(N, np.float32), wd=f32(wd))
    orc = OA.Tensor(p=p0.copy(), g=None, m=np.zeros(N, np.float32), v=np.zeros(N, np.float32), wd=f32(wd))
    ref = OA.Tensor(p=p0.astype(np.float64), g=None, m=np.zeros(N), v=np.zeros(N), wd=f32(wd))
    failures = []
    first_gap = None
    for t in range(1, steps + 1):
        g = rng.normal(0, 1e-3, N).astype(np.float32)
        orc.g, ref.g = g, g.astype(np.float64)
        s = OA.f32_scalars(lr=f32(lr), beta1=B1, beta2=B2, eps=EPS, t=t)
        got.p[...], got.m[...], got.v[...] = OA.elementwise_f32(
            got.p, g, got.m, got.v, s, OA.decay_f32(s.lr, got.wd), decay_after=decay_after)
        OA.step_f32([orc], lr=f32(lr), beta1=B1, beta2=B2, eps=EPS, t=t)
        OA.step_fp64([ref], lr=f32(lr), beta1=B1, beta2=B2, eps=EPS, t=t)
        checks = [("bit-exact", lambda: assert_state_bitexact(
            {"p": got.p, "m": got.m, "v": got.v}, {"p": orc.p, "m": orc.m, "v": orc.v}))]
        if t == 1:
            first_gap = float(np.max(np.abs(got.p.astype(np.float64) - ref.p)))
            checks.append(("single step", lambda: assert_single_step_rel(got.p, ref.p)))
        if t == steps:
            checks.append(("ten steps", lambda: assert_max_abs(got.p, ref.p)))
        for name, check in checks:
            try:
                check()
            except AssertionError:
                failures.append((t, name))
    return failures, first_gap


def test_decay_after_is_rejected_by_every_check():
    failures, gap = _run(wd=0.1, decay_after=True)
    names = {name for _, name in failures}
    assert names == {"bit-exact", "single step", "ten steps"}, failures
    assert (1, "bit-exact") in failures
    # the first-step gap is lr*wd*|lr*u| with |u| close to 1 from zero state
    assert 0.9e-3 < gap < 1.01e-3, gap


def test_orderings_agree_and_pass_at_zero_weight_decay():
    failures, gap = _run(wd=0.0, decay_after=True)
    assert failures == []
    assert gap < 1e-7


def test_the_correct_ordering_passes():
    failures, _ = _run(wd=0.1, decay_after=False, steps=3)
    assert failures == []


@pytest.mark.parametrize("wd", [0.1, 0.0])
def test_gap_is_lr_wd_times_the_step(wd):
    """At step one, from zero state, the two orderings differ by exactly
    fl32(lr*wd) * |fl32(step_size*u)| up to the float32 roundings of each side
    (at wd = 0 they are the same float32 operations)."""
    rng = np.random.default_rng(5)
    n = 4096
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    s = OA.f32_scalars(lr=f32(0.1), beta1=B1, beta2=B2, eps=EPS, t=1)
    d = OA.decay_f32(s.lr, f32(wd))
    z = np.zeros(n, np.float32)
    a, _, _ = OA.elementwise_f32(p, g, z, z, s, d)
    b, _, _ = OA.elementwise_f32(p, g, z, z, s, d, decay_after=True)
    step = np.abs((p.astype(np.float64) * np.float64(d)) - a.astype(np.float64))
    expect = (1.0 - np.float64(d)) * step
    # each side rounds p twice (within about one ulp of |p| <= 0.25, 1.5e-8 each)
    assert np.allclose(np.abs(a.astype(np.float64) - b), expect, rtol=0, atol=3e-8)
