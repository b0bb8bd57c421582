"""Shared helpers for the GPU parity tests: host <-> device copies and dtype views.

Inputs are generated on the host from seeded numpy generators (or, for the
full-size workloads, on the device by ``synth``), copied to the device for the
library and handed to the oracle as numpy arrays.  Nothing the oracle receives
comes out of the library.
"""

from __future__ import annotations

import numpy as np
import torch

F32 = np.float32


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.detach().cpu().numpy()


def bf16_bits(t_bf16: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor."""
    return t_bf16.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(F32)


def grads_of(x32: np.ndarray, dtype) -> tuple[torch.Tensor, np.ndarray]:
    """A grad tensor on the device in ``dtype`` and its exact float32 widening for the oracle."""
    if dtype == torch.float32:
        return dev(x32.astype(F32)), x32.astype(F32)
    if dtype == torch.float16:
        h = x32.astype(np.float16)
        return dev(h), h.astype(F32)
    t = torch.from_numpy(x32.astype(F32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    return t.cuda(), widen_bf16(bits)


def scalar_f32(x: float) -> torch.Tensor:
    return torch.tensor([x], dtype=torch.float32, device="cuda")


def scalar_i32(x: int) -> torch.Tensor:
    return torch.tensor([x], dtype=torch.int32, device="cuda")


def bits_equal(a, b) -> bool:
    a = np.asarray(a)
    b = np.asarray(b)
    if a.dtype == F32:
        a = a.view(np.uint32)
    if b.dtype == F32:
        b = b.view(np.uint32)
    return a.shape == b.shape and np.array_equal(a, b)


def first_mismatch(a, b) -> str:
    a = np.asarray(a, dtype=F32).ravel()
    b = np.asarray(b, dtype=F32).ravel()
    bad = np.nonzero(a.view(np.uint32) != b.view(np.uint32))[0]
    if bad.size == 0:
        return "identical"
    i = bad[0]
    return f"{bad.size} mismatches; first at {i}: gpu={a[i]!r} oracle={b[i]!r}"


# ---------------------------------------------------------------- acceptance checks
# The checks the GPU parity tests apply to the library's output.  They take
# numpy arrays, so that a CPU test can feed them a planted mistake (computed by
# the oracle) and show that they reject it.

def assert_state_bitexact(got: dict, want: dict, where: str = "") -> None:
    """Every named array of `got` bit-identical to the same name in `want`."""
    for k in want:
        assert bits_equal(got[k], want[k]), f"{where}{k}: {first_mismatch(got[k], want[k])}"


def assert_single_step_rel(p_got, p_fp64, tol: float = 1e-6) -> None:
    """One step against the float64 definition: |dp| within tol relative to the
    size of the terms (|p| plus the step of about lr = 0.1 at the workload)."""
    d = np.abs(np.asarray(p_got).astype(np.float64) - p_fp64)
    worst = float(np.max(d / (np.abs(p_fp64) + 0.1)))
    assert worst < tol, f"single step: {worst:.3e} relative to the float64 definition"


def assert_max_abs(p_got, p_fp64, tol: float = 5e-5) -> None:
    """Many steps against the float64 definition: max |dp| <= tol."""
    worst = float(np.max(np.abs(np.asarray(p_got).astype(np.float64) - p_fp64)))
    assert worst <= tol, f"max |dp| {worst:.3e} against the float64 definition"
