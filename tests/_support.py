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


# ---------------------------------------------------------------- guard bands
# Every device array a GPU parity test hands to the library sits inside a
# buffer with GUARD bytes of a fixed pseudo-random pattern before and after
# it (the payload itself starts as that pattern too, until the test fills
# it).  A store outside an array's bounds -- past a ragged tail, a lone 4-bit
# nibble, a partial 8-bit block, a misaligned view's first element -- lands in
# a band; ``assert_guards_intact`` reads every band back after a step, and a
# fixture in conftest.py checks them again at the end of every GPU test.
GUARD = 256
_PATTERN = np.random.default_rng(0x5EED_BA5D).integers(0, 256, 1 << 16, dtype=np.uint8)
_GUARDED: list = []      # (buffer, payload start byte, payload end byte)
DEVICE = "cuda"          # where guarded arrays live (the CPU test of the bands uses "cpu")


def _pattern(nbytes: int) -> np.ndarray:
    return np.resize(_PATTERN, nbytes)


def guarded_empty(n: int, dtype, shift: int = 0) -> torch.Tensor:
    """n elements of dtype on the device, between two guard bands; the array
    starts `shift` elements past a 256-byte boundary (shift > 0: a view off the
    16-byte grid)."""
    el = torch.empty(0, dtype=dtype).element_size()
    start = GUARD + shift * el
    end = start + n * el
    total = end + GUARD
    buf = torch.from_numpy(_pattern(total)).to(DEVICE)
    _GUARDED.append((buf, start, end))
    return buf[start:end].view(dtype)


def guards_reset() -> None:
    _GUARDED.clear()


def assert_guards_intact() -> None:
    """Every guard band of every array made since the last reset still holds its pattern."""
    if not _GUARDED:
        return
    bands = torch.cat([torch.cat([b[:s], b[e:]]) for b, s, e in _GUARDED]).cpu().numpy()
    want = np.concatenate([np.concatenate([_pattern(b.numel())[:s], _pattern(b.numel())[e:]])
                           for b, s, e in _GUARDED])
    if not np.array_equal(bands, want):
        off = 0
        for k, (b, s, e) in enumerate(_GUARDED):
            n = s + b.numel() - e
            if not np.array_equal(bands[off:off + n], want[off:off + n]):
                bad = np.nonzero(bands[off:off + n] != want[off:off + n])[0]
                where = [f"{int(i) - s} before the start" if i < s else f"{int(i) - s} past the end"
                         for i in bad[:4]]
                raise AssertionError(f"guard band of array {k} ({e - s} bytes) overwritten: "
                                     f"bytes {where}")
            off += n


def dev(a: np.ndarray, shift: int = 0) -> torch.Tensor:
    """A guarded device copy of a host array (see guarded_empty)."""
    a = np.ascontiguousarray(a)
    t = guarded_empty(a.size, torch.from_numpy(a[:0].copy()).dtype, shift)
    if a.size:
        t.copy_(torch.from_numpy(a.reshape(-1)))
    return t.view(a.shape) if a.ndim > 1 else t


def empty(n: int, dtype=torch.float32, shift: int = 0) -> torch.Tensor:
    """A guarded device array whose contents are the pattern until written."""
    return guarded_empty(n, dtype, shift)


def zeros(n: int, dtype=torch.float32, shift: int = 0) -> torch.Tensor:
    t = guarded_empty(n, dtype, shift)
    t.zero_()
    return t


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


def to_dev(t: torch.Tensor) -> torch.Tensor:
    """A guarded device copy of a host torch tensor."""
    out = guarded_empty(t.numel(), t.dtype)
    if t.numel():
        out.copy_(t.reshape(-1))
    return out


def scalar_f32(x: float) -> torch.Tensor:
    t = guarded_empty(1, torch.float32)
    t.fill_(x)
    return t


def scalar_i32(x: int) -> torch.Tensor:
    t = guarded_empty(1, torch.int32)
    t.fill_(x)
    return t


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
    return (f"{bad.size} mismatches; first at {i}: gpu={a[i]!r} oracle={b[i]!r}; "
            f"at {bad[:16].tolist()}")


# ---------------------------------------------------------------- acceptance checks
# The checks the GPU parity tests apply to the library's output.  They take
# numpy arrays, so that a CPU test can feed them a planted mistake (computed by
# the oracle) and show that they reject it.

def assert_state_bitexact(got: dict, want: dict, where: str = "", prev: dict | None = None) -> None:
    """Every named array of `got` bit-identical to the same name in `want`.  On a
    mismatch every array is reported, and with `prev` (the oracle's state one step
    earlier) how many of the mismatching values are exactly that earlier state --
    a step that was not applied there."""
    report = []
    for k in want:
        if not bits_equal(got[k], want[k]):
            msg = f"{where}{k}: {first_mismatch(got[k], want[k])}"
            if prev is not None and k in prev:
                g = np.asarray(got[k], dtype=F32).ravel()
                w = np.asarray(want[k], dtype=F32).ravel()
                bad = np.nonzero(g.view(np.uint32) != w.view(np.uint32))[0]
                old = np.asarray(prev[k], dtype=F32).ravel()[bad]
                same = int(np.sum(g[bad].view(np.uint32) == old.view(np.uint32)))
                msg += f"; {same} of {bad.size} equal the previous step's oracle value"
            report.append(msg)
    assert not report, " | ".join(report)


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
