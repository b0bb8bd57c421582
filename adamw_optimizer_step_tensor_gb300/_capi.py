"""ctypes binding of libadamw (include/adamw.h): argument marshalling only.

Every function here has the name and argument order of the C entry point it
wraps; pointers are passed as Python ints (``tensor.data_ptr()``) and the
stream as an int handle (``torch.cuda.current_stream().cuda_stream``).  A
non-OK status raises ``AdamWError`` carrying the library's message.  All
device work happens inside the library's kernels; nothing here computes.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libadamw.so")

OK, EINVAL, EALIGN, EDTYPE, ENOMEM, ECUDA, EUNSUPPORTED, ETIMEOUT = range(8)
STATUS_NAMES = ["OK", "EINVAL", "EALIGN", "EDTYPE", "ENOMEM", "ECUDA", "EUNSUPPORTED", "ETIMEOUT"]
F32, F16, BF16 = 0, 1, 2
MODE_FP32, MODE_BF16_REM, MODE_Q8, MODE_Q4 = 0, 1, 2, 3
Q8_BLOCK = 256
Q4_BLOCK = 128

_vp = ctypes.c_void_p


class AdamWError(RuntimeError):
    def __init__(self, status: int, message: str):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"ADAMW_{name}: {message}")
        self.status = status


class adamw_tensor(ctypes.Structure):
    _fields_ = [
        ("param", _vp),
        ("param_rem", _vp),
        ("grad", _vp),
        ("exp_avg", _vp),
        ("exp_avg_sq", _vp),
        ("absmax_m", _vp),
        ("absmax_v", _vp),
        ("numel", ctypes.c_int64),
        ("weight_decay", ctypes.c_float),
        ("exp_avg_slow", _vp),
    ]


_SIGNATURES = {
    "adamw_plan_create": (ctypes.c_int, [ctypes.POINTER(adamw_tensor), ctypes.c_int32, ctypes.c_int,
                                         ctypes.c_int, ctypes.POINTER(_vp)]),
    "adamw_mini_plan_create": (ctypes.c_int, [ctypes.POINTER(adamw_tensor), ctypes.POINTER(ctypes.c_int64),
                                              ctypes.c_int32, ctypes.c_int, ctypes.c_int,
                                              ctypes.POINTER(_vp)]),
    "adamw_mini_step": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                       _vp, _vp, _vp]),
    "adamw_plan_destroy": (ctypes.c_int, [_vp]),
    "adamw_plan_info": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int32)]),
    "adamw_plan_status": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "adamw_wait_selftest": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_double), _vp]),
    "adamw_check_nonfinite": (ctypes.c_int, [_vp, _vp, _vp]),
    "adamw_step": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                  _vp, _vp, _vp]),
    "adamw_step_noalloc": (ctypes.c_int, [ctypes.POINTER(adamw_tensor), ctypes.c_int32, ctypes.c_int,
                                          ctypes.c_int, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                          ctypes.c_float, _vp, _vp, _vp]),
    "adamw_step_noalloc_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "adamw_lr_from_table": (ctypes.c_int, [_vp, ctypes.c_int32, _vp, _vp, _vp]),
    "adamw_ademamix_step": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                           _vp, _vp, _vp]),
    "adamw_step_amp": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                      _vp, _vp, _vp]),
    "adamw_lion_step": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float, _vp, _vp, _vp]),
    "adamw_coupled_step": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                          _vp, _vp, _vp]),
    "adamw_bf16rem_split": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int64, _vp]),
    "adamw_bf16rem_join": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int64, _vp]),
    "adamw_q4_default_maps": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float),
                                             ctypes.POINTER(ctypes.c_float)]),
    "adamw_q8_default_maps": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float),
                                             ctypes.POINTER(ctypes.c_float)]),
    "adamw_q8_set_maps": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_float),
                                         ctypes.POINTER(ctypes.c_float)]),
    "adamw_q8_dequant": (ctypes.c_int, [_vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int64, _vp]),
    "adamw_q4_dequant": (ctypes.c_int, [_vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int64, _vp]),
    "adamw_q4_quant": (ctypes.c_int, [_vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int64, _vp]),
    "adamw_q8_quant": (ctypes.c_int, [_vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int64, _vp]),
    "adamw_last_error": (ctypes.c_char_p, []),
    "adamw_abi_version": (ctypes.c_int32, []),
}

_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library once (``path``, else $ADAMW_LIB, else the in-tree build);
    fails loudly when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("ADAMW_LIB") or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"libadamw.so not found at {path}; build it first with "
            "`python -m adamw_optimizer_step_tensor_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != OK:
        raise AdamWError(status, load().adamw_last_error().decode())


def adamw_last_error() -> str:
    return load().adamw_last_error().decode()


def adamw_abi_version() -> int:
    return int(load().adamw_abi_version())


def adamw_plan_create(tensors: list[adamw_tensor], mode: int, grad_dtype: int) -> int:
    arr = (adamw_tensor * max(1, len(tensors)))(*tensors)
    out = _vp()
    _check(load().adamw_plan_create(arr, len(tensors), mode, grad_dtype, ctypes.byref(out)))
    return out.value


def adamw_mini_plan_create(tensors: list[adamw_tensor], v_block: list[int], mode: int,
                           grad_dtype: int) -> int:
    arr = (adamw_tensor * max(1, len(tensors)))(*tensors)
    blocks = (ctypes.c_int64 * max(1, len(v_block)))(*v_block)
    out = _vp()
    _check(load().adamw_mini_plan_create(arr, blocks if v_block else None, len(tensors), mode,
                                         grad_dtype, ctypes.byref(out)))
    return out.value


def adamw_mini_step(plan: int, lr_dev: int, step_dev: int, beta1: float, beta2: float, eps: float,
                    grad_scale_dev: int | None, found_inf_dev: int | None, stream: int | None) -> None:
    _check(load().adamw_mini_step(plan, lr_dev, step_dev, beta1, beta2, eps, grad_scale_dev,
                                  found_inf_dev, stream))


def adamw_plan_destroy(plan: int) -> None:
    _check(load().adamw_plan_destroy(plan))


def adamw_plan_info(plan: int) -> dict:
    n, c = ctypes.c_int64(), ctypes.c_int64()
    g, b = ctypes.c_int32(), ctypes.c_int32()
    _check(load().adamw_plan_info(plan, ctypes.byref(n), ctypes.byref(c), ctypes.byref(g),
                                  ctypes.byref(b)))
    return {"total_numel": n.value, "n_chunks": c.value, "grid_blocks": g.value,
            "block_threads": b.value}


def adamw_plan_status(plan: int) -> int:
    """Fault bits of the plan's device-side pipeline; raises AdamWError (ETIMEOUT) if set."""
    bits = ctypes.c_uint32()
    _check(load().adamw_plan_status(plan, ctypes.byref(bits)))
    return bits.value


def adamw_wait_selftest(limit_us: int, stream: int | None) -> tuple[int, float]:
    """(status, ms waited) of the bounded-wait self-test; ETIMEOUT is its normal status."""
    ms = ctypes.c_double()
    st = load().adamw_wait_selftest(limit_us, ctypes.byref(ms), stream)
    if st not in (OK, ETIMEOUT):
        _check(st)
    return st, ms.value


def adamw_check_nonfinite(plan: int, found_inf_dev: int, stream: int | None) -> None:
    _check(load().adamw_check_nonfinite(plan, found_inf_dev, stream))


def adamw_step(plan: int, lr_dev: int, step_dev: int, beta1: float, beta2: float, eps: float,
               grad_scale_dev: int | None, found_inf_dev: int | None, stream: int | None) -> None:
    _check(load().adamw_step(plan, lr_dev, step_dev, beta1, beta2, eps, grad_scale_dev,
                             found_inf_dev, stream))


def adamw_step_noalloc(tensors: list[adamw_tensor], mode: int, grad_dtype: int, lr_dev: int,
                       step_dev: int, beta1: float, beta2: float, eps: float,
                       grad_scale_dev: int | None, found_inf_dev: int | None,
                       stream: int | None) -> None:
    """One step without allocating: for callers that cannot call cudaMalloc
    and so cannot build a plan (see include/adamw.h for limits and rules)."""
    arr = (adamw_tensor * max(1, len(tensors)))(*tensors)
    _check(load().adamw_step_noalloc(arr, len(tensors), mode, grad_dtype, lr_dev, step_dev, beta1,
                                     beta2, eps, grad_scale_dev, found_inf_dev, stream))


def adamw_step_noalloc_status() -> int:
    """Fault bits of adamw_step_noalloc's static array on the current device
    (read, then cleared); raises AdamWError (ETIMEOUT) if any was set."""
    bits = ctypes.c_uint32()
    _check(load().adamw_step_noalloc_status(ctypes.byref(bits)))
    return bits.value


def adamw_ademamix_step(plan: int, lr_dev: int, step_dev: int, beta1: float, beta2: float,
                        beta3: float, alpha: float, eps: float, grad_scale_dev: int | None,
                        found_inf_dev: int | None, stream: int | None) -> None:
    _check(load().adamw_ademamix_step(plan, lr_dev, step_dev, beta1, beta2, beta3, alpha, eps,
                                      grad_scale_dev, found_inf_dev, stream))


def adamw_lion_step(plan: int, lr_dev: int, step_dev: int, beta1: float, beta2: float,
                    grad_scale_dev: int | None, found_inf_dev: int | None, stream: int | None) -> None:
    _check(load().adamw_lion_step(plan, lr_dev, step_dev, beta1, beta2, grad_scale_dev,
                                  found_inf_dev, stream))


RULES = {"momentum": 0, "rmsprop": 1, "adagrad": 2}


def adamw_coupled_step(plan: int, rule: int, lr_dev: int, step_dev: int, beta: float, eps: float,
                       grad_scale_dev: int | None, found_inf_dev: int | None,
                       stream: int | None) -> None:
    _check(load().adamw_coupled_step(plan, rule, lr_dev, step_dev, beta, eps, grad_scale_dev,
                                     found_inf_dev, stream))


def adamw_step_amp(plan: int, lr_dev: int, step_dev: int, beta1: float, beta2: float, eps: float,
                   grad_scale_dev: int | None, found_inf_dev: int, stream: int | None) -> None:
    _check(load().adamw_step_amp(plan, lr_dev, step_dev, beta1, beta2, eps, grad_scale_dev,
                                 found_inf_dev, stream))


def adamw_lr_from_table(table: int, n: int, step_dev: int, lr_dev: int, stream: int | None) -> None:
    _check(load().adamw_lr_from_table(table, n, step_dev, lr_dev, stream))


def adamw_bf16rem_split(master: int, bf16: int, rem: int, n: int, stream: int | None) -> None:
    _check(load().adamw_bf16rem_split(master, bf16, rem, n, stream))


def adamw_bf16rem_join(bf16: int, rem: int, master: int, n: int, stream: int | None) -> None:
    _check(load().adamw_bf16rem_join(bf16, rem, master, n, stream))


def adamw_q4_default_maps():
    """Host call: returns (signed_map, unsigned_map) of the Q4 mode, two lists of 16 floats."""
    s, u = (ctypes.c_float * 16)(), (ctypes.c_float * 16)()
    _check(load().adamw_q4_default_maps(s, u))
    return list(s), list(u)


def adamw_q8_default_maps():
    """Host call: returns (signed_map, unsigned_map) as two lists of 256 floats."""
    s, u = (ctypes.c_float * 256)(), (ctypes.c_float * 256)()
    _check(load().adamw_q8_default_maps(s, u))
    return list(s), list(u)


def adamw_q8_set_maps(plan: int, signed_map, unsigned_map) -> None:
    s = (ctypes.c_float * 256)(*[float(x) for x in signed_map])
    u = (ctypes.c_float * 256)(*[float(x) for x in unsigned_map])
    _check(load().adamw_q8_set_maps(plan, s, u))


def adamw_q8_dequant(plan: int, which: int, codes: int, absmax: int, out: int, n: int,
                     stream: int | None) -> None:
    _check(load().adamw_q8_dequant(plan, which, codes, absmax, out, n, stream))


def adamw_q8_quant(plan: int, which: int, x: int, codes: int, absmax: int, n: int,
                   stream: int | None) -> None:
    _check(load().adamw_q8_quant(plan, which, x, codes, absmax, n, stream))


def adamw_q4_dequant(plan: int, which: int, codes: int, absmax: int, out: int, n: int,
                     stream: int | None) -> None:
    _check(load().adamw_q4_dequant(plan, which, codes, absmax, out, n, stream))


def adamw_q4_quant(plan: int, which: int, x: int, codes: int, absmax: int, n: int,
                   stream: int | None) -> None:
    _check(load().adamw_q4_quant(plan, which, x, codes, absmax, n, stream))
