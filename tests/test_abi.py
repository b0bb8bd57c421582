"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, validates arguments on the host before any CUDA call, and its
host-side default code maps equal the oracle's bit for bit."""

import ctypes
import os
import re

import numpy as np
import pytest

from adamw_optimizer_step_tensor_gb300 import _capi as C
from oracle import qmap

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "adamw.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[a-z_0-9 ]*?\**\s*\b(adamw_[a-z0-9_]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("adamw_plan_create", "adamw_step", "adamw_check_nonfinite", "adamw_bf16rem_split",
              "adamw_bf16rem_join", "adamw_q8_set_maps", "adamw_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = C.load()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_wraps_every_declared_symbol():
    for name in declared_functions():
        assert callable(getattr(C, name)), name


def test_abi_version():
    assert C.adamw_abi_version() == 3


def test_default_maps_equal_oracle_maps():
    s, u = C.adamw_q8_default_maps()
    s = np.array(s, np.float32)
    u = np.array(u, np.float32)
    assert np.array_equal(s.view(np.uint32), qmap.signed_map().view(np.uint32))
    assert np.array_equal(u.view(np.uint32), qmap.unsigned_map().view(np.uint32))


def _t(base=0x10000, numel=1024, rem=None, am=None, av=None, wd=0.0):
    return C.adamw_tensor(base, rem, base + 0x100000, base + 0x200000, base + 0x300000,
                          am, av, numel, wd)


def _status(fn):
    with pytest.raises(C.AdamWError) as e:
        fn()
    return e.value.status


def test_plan_create_rejects_bad_arguments_on_the_host():
    assert _status(lambda: C.adamw_plan_create([], 9, C.F32)) == C.EDTYPE
    assert _status(lambda: C.adamw_plan_create([], C.MODE_FP32, 7)) == C.EDTYPE
    assert _status(lambda: C.adamw_plan_create([_t(numel=-1)], C.MODE_FP32, C.F32)) == C.EINVAL
    assert _status(lambda: C.adamw_plan_create([_t(base=0x10002)], C.MODE_FP32, C.F32)) == C.EALIGN
    # remainder pointer only in BF16_REM mode; absmax only in Q8 mode
    assert _status(lambda: C.adamw_plan_create([_t(rem=0x900000)], C.MODE_FP32, C.F32)) == C.EINVAL
    assert _status(lambda: C.adamw_plan_create([_t()], C.MODE_BF16_REM, C.BF16)) == C.EINVAL
    assert _status(lambda: C.adamw_plan_create([_t()], C.MODE_Q8, C.BF16)) == C.EINVAL
    assert _status(lambda: C.adamw_plan_create([_t(wd=float("nan"))], C.MODE_FP32, C.F32)) == C.EINVAL
    missing = C.adamw_tensor(None, None, 0x1000, 0x2000, 0x3000, None, None, 16, 0.0)
    assert _status(lambda: C.adamw_plan_create([missing], C.MODE_FP32, C.F32)) == C.EINVAL
    assert "param" in C.adamw_last_error()


def test_negative_count_rejected():
    lib = C.load()
    out = ctypes.c_void_p()
    assert lib.adamw_plan_create(None, -1, 0, 0, ctypes.byref(out)) == C.EINVAL


def test_step_and_helpers_reject_bad_arguments_on_the_host():
    assert _status(lambda: C.adamw_step(None, 0x100, 0x200, 0.9, 0.999, 1e-8, None, None, None)) == C.EINVAL
    assert _status(lambda: C.adamw_check_nonfinite(None, 0x100, None)) == C.EINVAL
    assert _status(lambda: C.adamw_bf16rem_split(0x100, 0x200, 0x300, -1, None)) == C.EINVAL
    assert _status(lambda: C.adamw_bf16rem_join(0x100, 0x201, 0x300, 5, None)) == C.EALIGN
    assert _status(lambda: C.adamw_q8_dequant(None, 0, 0x100, 0x200, 0x300, 5, None)) == C.EINVAL
    # nothing to do: no launch, no error
    C.adamw_bf16rem_split(None, None, None, 0, None)
    C.adamw_bf16rem_join(None, None, None, 0, None)


def test_plan_info_null():
    assert _status(lambda: C.adamw_plan_info(None)) == C.EINVAL


def test_one_state_plans_are_checked_on_the_host():
    no_v = C.adamw_tensor(0x10000, None, 0x110000, 0x210000, None, None, None, 1024, 0.0)
    # exp_avg_sq on some tensors but not all
    assert _status(lambda: C.adamw_plan_create([no_v, _t(base=0x400000)], C.MODE_FP32, C.F32)) == C.EINVAL
    assert "exp_avg_sq" in C.adamw_last_error()
    # Q8 always needs v
    q = C.adamw_tensor(0x10000, None, 0x110000, 0x210000, None, 0x310000, 0x320000, 1024, 0.0)
    assert _status(lambda: C.adamw_plan_create([q], C.MODE_Q8, C.F32)) == C.EINVAL
    # AdEMAMix needs v
    slow = C.adamw_tensor(0x10000, None, 0x110000, 0x210000, None, None, None, 1024, 0.0, 0x510000)
    assert _status(lambda: C.adamw_plan_create([slow], C.MODE_FP32, C.F32)) == C.EINVAL
    assert _status(lambda: C.adamw_lion_step(None, 0x100, 0x200, 0.9, 0.99, None, None, None)) == C.EINVAL


def test_coupled_step_checks_on_the_host():
    assert _status(lambda: C.adamw_coupled_step(None, 0, 0x100, 0x200, 0.9, 1e-8, None, None, None)) == C.EINVAL
    assert C.RULES == {"momentum": 0, "rmsprop": 1, "adagrad": 2}


def test_q4_default_maps_equal_oracle_maps():
    s, u = C.adamw_q4_default_maps()
    assert np.array_equal(np.array(s, np.float32).view(np.uint32), qmap.signed_map4().view(np.uint32))
    assert np.array_equal(np.array(u, np.float32).view(np.uint32), qmap.unsigned_map4().view(np.uint32))


def test_q4_plans_are_checked_on_the_host():
    # absmax pointers are required in Q4 mode, param_rem is not allowed
    assert _status(lambda: C.adamw_plan_create([_t()], C.MODE_Q4, C.BF16)) == C.EINVAL
    assert _status(lambda: C.adamw_plan_create([_t(rem=0x900000, am=0x910000, av=0x920000)],
                                               C.MODE_Q4, C.BF16)) == C.EINVAL
    assert _status(lambda: C.adamw_plan_create([_t()], 4, C.BF16)) == C.EDTYPE


def test_mini_plans_are_checked_on_the_host():
    t = _t(numel=1024)
    assert _status(lambda: C.adamw_mini_plan_create([t], [3], C.MODE_FP32, C.F32)) == C.EINVAL   # 3 does not divide
    assert _status(lambda: C.adamw_mini_plan_create([t], [4], C.MODE_FP32, C.F32)) == C.EINVAL   # not a multiple of 8
    assert _status(lambda: C.adamw_mini_plan_create([t], [0], C.MODE_FP32, C.F32)) == C.EINVAL
    q = _t(numel=1024, am=0x910000, av=0x920000)
    assert _status(lambda: C.adamw_mini_plan_create([q], [256], C.MODE_Q8, C.F32)) == C.EUNSUPPORTED
    no_v = C.adamw_tensor(0x10000, None, 0x110000, 0x210000, None, None, None, 1024, 0.0)
    assert _status(lambda: C.adamw_mini_plan_create([no_v], [1024], C.MODE_FP32, C.F32)) == C.EINVAL
    assert _status(lambda: C.adamw_mini_step(None, 0x100, 0x200, 0.9, 0.999, 1e-8, None, None, None)) == C.EINVAL


def test_q4_io_checks_on_the_host():
    assert _status(lambda: C.adamw_q4_dequant(None, 0, 0x100, 0x200, 0x300, 5, None)) == C.EINVAL
    assert _status(lambda: C.adamw_q4_quant(None, 0, 0x100, 0x200, 0x300, 5, None)) == C.EINVAL
