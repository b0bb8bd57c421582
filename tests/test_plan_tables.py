"""The tables a plan builds and the launch shapes it asks for (CPU only).

The plan code of libadamw (``capi.cpp``, ``qmap.cpp``) is compiled for the host
and linked against ``tests/host/fake_runtime.cpp``: a fake CUDA runtime whose
"device" memory is host memory and recording stand-ins for the kernel
launchers (the SM count is 152, one bulk CTA per SM, one 1024-thread 8-bit
CTA, four 4-bit CTAs, two RMSprop/Adagrad CTAs).  The tests create plans
through the real entry points with fake tensor addresses, take a step, and
read back what the kernel would have been given: every tensor is cut into
chunks of the documented size that cover it once, in order; the grid is the
chunk count capped at the resident CTAs; the tensor table holds the caller's
pointers, sizes, decays and the 16-byte alignment flag; Adam-mini chunks never
straddle a shared-v block and the block table and reduction list agree with
them; the fused AMP step gets its own table; plan_info reports the CTA size.
"""

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

from adamw_optimizer_step_tensor_gb300 import _capi as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "adamw_optimizer_step_tensor_gb300", "csrc")
SMS = 152
CHUNK = np.dtype([("start", "<i8"), ("tensor", "<i4"), ("len", "<i4")])
TDESC = np.dtype([("p", "<u8"), ("rem", "<u8"), ("g", "<u8"), ("m", "<u8"), ("v", "<u8"),
                  ("am", "<u8"), ("av", "<u8"), ("m2", "<u8"), ("numel", "<i8"), ("wd", "<f4"),
                  ("vec_ok", "<i4")])
BLOCK = np.dtype([("v_index", "<i8"), ("first_chunk", "<i8"), ("len", "<i8"), ("tensor", "<i4"),
                  ("n_chunks", "<i4")])
_vp = ctypes.c_void_p


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            return os.path.join(d, "include")
    return None


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    so = tmp_path_factory.mktemp("host") / "libadamw_host.so"
    # -Bsymbolic: the plan code must call this library's fake runtime even when
    # the process has the real one loaded (torch)
    subprocess.run([cxx, "-std=c++17", "-O1", "-shared", "-fPIC", "-Wl,-Bsymbolic",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", CSRC, "-I", inc, os.path.join(CSRC, "capi.cpp"), os.path.join(CSRC, "qmap.cpp"),
                    os.path.join(ROOT, "tests", "host", "fake_runtime.cpp"), "-o", str(so)],
                   check=True, capture_output=True)
    L = ctypes.CDLL(str(so))
    sig = {
        "adamw_plan_create": (ctypes.c_int, [ctypes.POINTER(C.adamw_tensor), ctypes.c_int32,
                                             ctypes.c_int, ctypes.c_int, ctypes.POINTER(_vp)]),
        "adamw_mini_plan_create": (ctypes.c_int, [ctypes.POINTER(C.adamw_tensor),
                                                  ctypes.POINTER(ctypes.c_int64), ctypes.c_int32,
                                                  ctypes.c_int, ctypes.c_int, ctypes.POINTER(_vp)]),
        "adamw_plan_destroy": (ctypes.c_int, [_vp]),
        "adamw_plan_info": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int64),
                                           ctypes.POINTER(ctypes.c_int64),
                                           ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
        "adamw_step": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                      _vp, _vp, _vp]),
        "adamw_step_amp": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                          ctypes.c_float, _vp, _vp, _vp]),
        "adamw_mini_step": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_float, _vp, _vp, _vp]),
        "adamw_coupled_step": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp, ctypes.c_float,
                                              ctypes.c_float, _vp, _vp, _vp]),
        "adamw_last_error": (ctypes.c_char_p, []),
        "probe_kind": (ctypes.c_char_p, [ctypes.c_int]),
        "probe_grid": (ctypes.c_int, [ctypes.c_int]),
        "probe_algo": (ctypes.c_int, [ctypes.c_int]),
        "probe_tensors": (_vp, [ctypes.c_int]),
        "probe_chunks": (_vp, [ctypes.c_int]),
        "probe_n_chunks": (ctypes.c_int64, [ctypes.c_int]),
        "probe_chunk_blk": (_vp, [ctypes.c_int]),
        "probe_blocks": (_vp, [ctypes.c_int]),
        "probe_red_chunks": (_vp, [ctypes.c_int]),
        "probe_n_red": (ctypes.c_int64, [ctypes.c_int]),
        "probe_set_sms": (None, [ctypes.c_int]),
        "probe_small_args": (_vp, []),
        "probe_small_smem": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    L.probe_set_sms(SMS)
    return L


def _read(ptr, dtype, n):
    if n == 0:
        return np.zeros(0, dtype)
    buf = (ctypes.c_char * (dtype.itemsize * n)).from_address(ptr)
    return np.frombuffer(bytes(buf), dtype=dtype, count=n)


def _choose_chunk(total, bps):
    resident = SMS * bps
    c = -(-total // resident)
    c = -(-c // 256) * 256
    return min(max(c, 256), 16384)


class Fake:
    """Fake device addresses: one 4 GiB window per tensor and array."""

    def __init__(self):
        self.next = 1 << 40

    def __call__(self, nbytes, misalign=0):
        a = self.next
        self.next += (nbytes // (1 << 32) + 1) << 32        # the next window, 4 GiB aligned
        return a + misalign


def _records(sizes, mode, fake, misalign=(), with_v=True):
    recs = []
    for i, n in enumerate(sizes):
        state = 1 if mode in (C.MODE_Q8, C.MODE_Q4) else 4
        codes = (n + 1) // 2 if mode == C.MODE_Q4 else n * state
        psz = 2 if mode == C.MODE_BF16_REM else 4
        blk = 128 if mode == C.MODE_Q4 else 256
        recs.append(C.adamw_tensor(
            fake(n * psz, 4 if i in misalign else 0),
            fake(n * 2) if mode == C.MODE_BF16_REM else None,
            fake(n * 2), fake(codes), fake(codes) if with_v else None,
            fake(-(-n // blk) * 4) if mode in (C.MODE_Q8, C.MODE_Q4) else None,
            fake(-(-n // blk) * 4) if mode in (C.MODE_Q8, C.MODE_Q4) else None,
            n, 0.1 * (i % 3), None))
    return recs


def _create(L, recs, mode, gdt=C.BF16, blocks=None):
    arr = (C.adamw_tensor * max(1, len(recs)))(*recs)
    plan = _vp()
    if blocks is None:
        st = L.adamw_plan_create(arr, len(recs), mode, gdt, ctypes.byref(plan))
    else:
        b = (ctypes.c_int64 * max(1, len(blocks)))(*blocks)
        st = L.adamw_mini_plan_create(arr, b, len(recs), mode, gdt, ctypes.byref(plan))
    assert st == C.OK, L.adamw_last_error()
    return plan


def _scalars(fake):
    return fake(4), fake(4)


def _check_cover(chunks, sizes, chunk, tensors_first=None):
    """Per tensor, in order: starts 0, chunk, 2*chunk, ..., lengths to the end."""
    k = 0
    for i, n in enumerate(sizes):
        for s in range(0, n, chunk):
            c = chunks[k]
            assert (c["tensor"], c["start"], c["len"]) == (i, s, min(chunk, n - s)), (i, s, c)
            k += 1
    assert k == len(chunks)


SIZES = [1, 255, 256, 257, 0, 70_001, 16_384, 16_385, 3_000_000, 5]


@pytest.mark.parametrize("mode,bps,kind", [(C.MODE_FP32, 1, "bulk"), (C.MODE_BF16_REM, 1, "bulk"),
                                          (C.MODE_Q8, 1, "step"), (C.MODE_Q4, 4, "q4")])
def test_chunk_table_covers_every_tensor(lib, mode, bps, kind):
    fake = Fake()
    recs = _records(SIZES, mode, fake, misalign=(2,))
    plan = _create(lib, recs, mode)
    try:
        lr, step = _scalars(fake)
        assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
        assert lib.probe_kind(0).decode() == kind
        n_chunks = lib.probe_n_chunks(0)
        chunks = _read(lib.probe_chunks(0), CHUNK, n_chunks)
        chunk = _choose_chunk(sum(SIZES), bps)
        _check_cover(chunks, SIZES, chunk)
        assert lib.probe_grid(0) == min(n_chunks, bps * SMS)
        tds = _read(lib.probe_tensors(0), TDESC, len(SIZES))
        for i, (r, t) in enumerate(zip(recs, tds)):
            assert t["numel"] == r.numel and t["wd"] == np.float32(r.weight_decay), i
            if r.numel == 0:
                continue                                        # empty tensors are ignored
            assert t["p"] == r.param and t["g"] == r.grad and t["m"] == r.exp_avg, i
            assert t["vec_ok"] == (0 if i == 2 else 1), i          # tensor 2's param is 4 bytes off
        n = ctypes.c_int64()
        nc = ctypes.c_int64()
        g = ctypes.c_int32()
        b = ctypes.c_int32()
        assert lib.adamw_plan_info(plan, ctypes.byref(n), ctypes.byref(nc), ctypes.byref(g),
                                   ctypes.byref(b)) == C.OK
        assert n.value == sum(SIZES) and nc.value == n_chunks and g.value == lib.probe_grid(0)
        assert b.value == {"bulk": 544, "step": 1024, "q4": 256}[kind]
    finally:
        lib.adamw_plan_destroy(plan)


def test_chunk_size_limits(lib):
    fake = Fake()
    for sizes, want in (([1000], 256), ([152 * 1000], 1024), ([1 << 30], 16384)):
        plan = _create(lib, _records(sizes, C.MODE_FP32, fake), C.MODE_FP32, C.F32)
        try:
            lr, step = _scalars(fake)
            # momentum walks the plan's chunk table whatever the plan's size
            assert lib.adamw_coupled_step(plan, C.RULES["momentum"], lr, step, 0.9, 1e-8, None,
                                          None, None) == C.OK
            chunks = _read(lib.probe_chunks(0), CHUNK, lib.probe_n_chunks(0))
            assert chunks[0]["len"] == min(want, sizes[0]), sizes
            _check_cover(chunks, sizes, want)
        finally:
            lib.adamw_plan_destroy(plan)


def test_sqrt_div_rules_take_two_ctas_per_sm(lib):
    fake = Fake()
    sizes = [10_000_000, 3]
    plan = _create(lib, _records(sizes, C.MODE_FP32, fake, with_v=False), C.MODE_FP32, C.F32)
    try:
        lr, step = _scalars(fake)
        n_chunks = None
        for rule, per_sm, algo in (("momentum", 1, 3), ("rmsprop", 2, 4), ("adagrad", 2, 5)):
            assert lib.adamw_coupled_step(plan, C.RULES[rule], lr, step, 0.9, 1e-8, None, None,
                                          None) == C.OK
            n_chunks = lib.probe_n_chunks(0)
            assert lib.probe_algo(0) == algo
            assert lib.probe_grid(0) == min(n_chunks, per_sm * SMS), rule
        # a 1-state plan refuses the two-state step
        assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.EINVAL
    finally:
        lib.adamw_plan_destroy(plan)


def test_adam_mini_chunks_stay_inside_blocks(lib):
    fake = Fake()
    sizes = [50_000, 64 * 12, 2048, 777, 3 * 40_000, 100_003, 16 * 300, 0, 4 * 70_000]
    blocks = [1, 64, 2048, 777, 40_000, 100_003, 16, 1, 70_000]
    plan = _create(lib, _records(sizes, C.MODE_FP32, fake), C.MODE_FP32, C.F32, blocks=blocks)
    try:
        lr, step = _scalars(fake)
        assert lib.adamw_mini_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
        assert lib.probe_kind(0).decode() == "bulk" and lib.probe_algo(0) == 6
        assert lib.probe_kind(1).decode() == "mini_reduce"
        n_chunks = lib.probe_n_chunks(0)
        chunks = _read(lib.probe_chunks(0), CHUNK, n_chunks)
        cblk = _read(lib.probe_chunk_blk(0), np.dtype("<i4"), n_chunks)
        n_red = lib.probe_n_red(1)
        red = _read(lib.probe_red_chunks(1), np.dtype("<i8"), n_red)
        n_blocks = sum(n // b for n, b in zip(sizes, blocks) if b > 1 and n > 0)
        blk = _read(lib.probe_blocks(1), BLOCK, n_blocks)
        chunk = _choose_chunk(sum(sizes), 1)
        k, bi = 0, 0
        for i, (n, b) in enumerate(zip(sizes, blocks)):
            if b == 1 or n == 0:
                for s in range(0, n, chunk):
                    assert (chunks[k]["tensor"], chunks[k]["start"]) == (i, s) and cblk[k] == -1
                    k += 1
                continue
            for b0 in range(0, n, b):
                B = blk[bi]
                assert (B["tensor"], B["v_index"], B["len"], B["first_chunk"]) == (i, b0 // b, b, k)
                assert B["n_chunks"] == -(-b // chunk)
                for s in range(0, b, chunk):
                    c = chunks[k]
                    assert (c["tensor"], c["start"], c["len"]) == (i, b0 + s, min(chunk, b - s))
                    assert cblk[k] == bi
                    k += 1
                bi += 1
        assert k == n_chunks and bi == n_blocks
        assert np.array_equal(red, np.flatnonzero(cblk >= 0))
    finally:
        lib.adamw_plan_destroy(plan)


def test_fused_amp_table_and_threshold(lib):
    fake = Fake()
    for sizes, fused in (([3 << 20, 4097], True), ([7 << 20], False)):
        plan = _create(lib, _records(sizes, C.MODE_FP32, fake), C.MODE_FP32, C.F16)
        try:
            lr, step = _scalars(fake)
            found = fake(4)
            assert lib.adamw_step_amp(plan, lr, step, 0.9, 0.999, 1e-8, fake(4), found, None) == C.OK
            if fused:
                assert lib.probe_kind(0).decode() == "fused_amp"
                n_chunks = lib.probe_n_chunks(0)
                chunks = _read(lib.probe_chunks(0), CHUNK, n_chunks)
                _check_cover(chunks, sizes, _choose_chunk(sum(sizes), 2))
                assert lib.probe_grid(0) == min(n_chunks, 2 * SMS)
            else:                       # above 6 Mi elements: check, then the bulk step
                assert lib.probe_kind(1).decode() == "nonfinite"
                assert lib.probe_kind(0).decode() == "bulk"
        finally:
            lib.adamw_plan_destroy(plan)


def _cluster_map(k):
    """A signed map with k extra levels 0.0008 apart just above 0.6: their
    thresholds crowd one bucket of the nearest-code search."""
    grid = np.linspace(-1, 1, 241)
    pads = (grid[12:12 + 15 - k] + grid[13:13 + 15 - k]) / 2
    return np.sort(np.concatenate([grid, 0.6 + 0.0008 * np.arange(1, k + 1), pads])).astype(np.float32)


def test_q8_maps_set_the_compares_per_lookup(lib):
    lib.adamw_q8_set_maps.restype = ctypes.c_int
    lib.adamw_q8_set_maps.argtypes = [_vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
    lib.probe_refine.restype, lib.probe_refine.argtypes = ctypes.c_int, [ctypes.c_int]
    fake = Fake()
    plan = _create(lib, _records([100_000], C.MODE_Q8, fake), C.MODE_Q8)
    try:
        lr, step = _scalars(fake)
        umap = np.linspace(0, 1, 256).astype(np.float32)
        fp = ctypes.POINTER(ctypes.c_float)
        assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
        assert lib.probe_refine(0) == 1                       # the default maps: one compare
        for k, refine in ((3, 2), (5, 3)):
            smap = _cluster_map(k)
            assert lib.adamw_q8_set_maps(plan, smap.ctypes.data_as(fp), umap.ctypes.data_as(fp)) == C.OK
            assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
            assert lib.probe_refine(0) == refine, k
        assert lib.adamw_q8_set_maps(plan, _cluster_map(7).ctypes.data_as(fp),
                                     umap.ctypes.data_as(fp)) == C.EUNSUPPORTED
        assert b"too dense" in lib.adamw_last_error()
        assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
        assert lib.probe_refine(0) == 3                       # a refused map leaves the plan as it was
    finally:
        lib.adamw_plan_destroy(plan)


def test_rule_launches_and_empty_plans(lib):
    lib.adamw_ademamix_step.restype = ctypes.c_int
    lib.adamw_ademamix_step.argtypes = [_vp, _vp, _vp] + [ctypes.c_float] * 5 + [_vp, _vp, _vp]
    lib.adamw_lion_step.restype = ctypes.c_int
    lib.adamw_lion_step.argtypes = [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float, _vp, _vp, _vp]
    fake = Fake()
    lr, step = _scalars(fake)
    # AdEMAMix: the slow EMA reaches the tensor table, the bulk kernel runs rule 1
    recs = _records([5000, 300], C.MODE_FP32, fake)
    for r in recs:
        r.exp_avg_slow = fake(r.numel * 4)
    plan = _create(lib, recs, C.MODE_FP32, C.F32)
    try:
        assert lib.adamw_ademamix_step(plan, lr, step, 0.9, 0.999, 0.9999, 5.0, 1e-8, None, None,
                                       None) == C.OK
        assert lib.probe_kind(0).decode() == "bulk" and lib.probe_algo(0) == 1
        tds = _read(lib.probe_tensors(0), TDESC, 2)
        assert [int(t["m2"]) for t in tds] == [r.exp_avg_slow for r in recs]
        # the same plan's AdamW step: a small plan, staged whole in shared memory
        assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
        assert lib.probe_kind(0).decode() == "small"
    finally:
        lib.adamw_plan_destroy(plan)
    # Lion on a 1-state plan: rule 2, one CTA per SM
    plan = _create(lib, _records([1 << 22], C.MODE_BF16_REM, fake, with_v=False), C.MODE_BF16_REM)
    try:
        assert lib.adamw_lion_step(plan, lr, step, 0.9, 0.99, None, None, None) == C.OK
        assert lib.probe_algo(0) == 2
        assert lib.probe_grid(0) == min(lib.probe_n_chunks(0), SMS)
        tds = _read(lib.probe_tensors(0), TDESC, 1)
        assert tds[0]["v"] == 0 and tds[0]["rem"] != 0
    finally:
        lib.adamw_plan_destroy(plan)
    # an empty plan still launches (one CTA, no chunks): the step counter advances on device
    for mode in (C.MODE_FP32, C.MODE_Q8, C.MODE_Q4):
        plan = _create(lib, [], mode)
        try:
            assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
            assert lib.probe_n_chunks(0) == 0 and lib.probe_grid(0) == 1, mode
        finally:
            lib.adamw_plan_destroy(plan)


SMALLT = np.dtype([("p", "<u8"), ("rem", "<u8"), ("g", "<u8"), ("m", "<u8"), ("v", "<u8"),
                   ("numel", "<i8"), ("wd", "<f4"), ("first_item", "<i4"), ("piece", "<i4"),
                   ("vec_ok", "<i4")], align=True)


def _small_args(lib):
    raw = _read(lib.probe_small_args(), np.dtype("u1"), 56 + 16 * SMALLT.itemsize).tobytes()
    n_tensors = int(np.frombuffer(raw[52:56], "<i4")[0])
    return n_tensors, np.frombuffer(raw[56:], SMALLT)[:n_tensors]


@pytest.mark.parametrize("mode,gdt,sizes", [
    (C.MODE_FP32, C.F32, [1 << 20]),
    (C.MODE_FP32, C.F16, [1 << 20, 4097]),
    (C.MODE_BF16_REM, C.BF16, [1000]),
    (C.MODE_FP32, C.BF16, [1, 3, 8, 9, 255, 256, 257, 2047, 2048, 2049, 8191, 8192, 8193, 50001, 0, 7]),
    (C.MODE_FP32, C.F32, [152 * 1000]),
])
def test_small_plans_stage_whole_pieces(lib, mode, gdt, sizes):
    """A small plan: every non-empty tensor in pieces of one length (a multiple of 8,
    at least 256), pieces numbered tensor by tensor, one CTA each, at most one per SM,
    and each CTA's 32 warp slices of one piece within 216 KB of shared memory; both
    adamw_step launches it, and adamw_step_amp its fused variant when every tensor is
    16-byte aligned."""
    fake = Fake()
    recs = _records(sizes, mode, fake, misalign=(1,) if len(sizes) > 2 else ())
    plan = _create(lib, recs, mode, gdt)
    try:
        lr, step = _scalars(fake)
        assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
        assert lib.probe_kind(0).decode() == "small"
        grid = lib.probe_grid(0)
        n, t = _small_args(lib)
        live = [(i, r) for i, r in enumerate(recs) if r.numel > 0]
        assert n == len(live)
        piece = int(t[0]["piece"])
        assert piece % 8 == 0 and piece >= 256 and all(int(x["piece"]) == piece for x in t)
        first = 0
        for (i, r), x in zip(live, t):
            assert x["numel"] == r.numel and x["p"] == r.param and x["g"] == r.grad, i
            assert x["m"] == r.exp_avg and x["v"] == r.exp_avg_sq and x["rem"] == (r.param_rem or 0), i
            assert x["wd"] == np.float32(r.weight_decay) and x["first_item"] == first, i
            assert x["vec_ok"] == (0 if (len(sizes) > 2 and i == 1) else 1), i
            first += -(-r.numel // piece)
        assert grid == first <= SMS
        per_elem = (4 if mode == C.MODE_FP32 else 4) + (2 if gdt != C.F32 else 4) + 8
        slice_ = -(-(piece // 8 * 8) // (32 * 8)) * 8          # 32 warps, slices of 8k elements
        assert lib.probe_small_smem() == max(16, 32 * slice_ * per_elem) <= 216 * 1024
        b = ctypes.c_int32()
        g = ctypes.c_int32()
        assert lib.adamw_plan_info(plan, None, None, ctypes.byref(g), ctypes.byref(b)) == C.OK
        assert (g.value, b.value) == (grid, 1024)
        found = fake(4)
        assert lib.adamw_step_amp(plan, lr, step, 0.9, 0.999, 1e-8, fake(4), found, None) == C.OK
        if len(sizes) > 2:
            # a tensor off the 16-byte grid: the fused check + step takes the chunked path
            assert lib.probe_kind(0).decode() == "fused_amp"
        else:
            # the fused variant stages its results beside the originals
            assert lib.probe_kind(0).decode() == "small_fused" and lib.probe_grid(0) == grid
            extra = (4 if mode == C.MODE_FP32 else 4) + 8
            assert lib.probe_small_smem() == max(16, 32 * slice_ * (per_elem + extra)) <= 216 * 1024
    finally:
        lib.adamw_plan_destroy(plan)


def test_plans_beyond_the_shared_memory_size_stay_on_the_bulk_path(lib):
    fake = Fake()
    for sizes, mode, gdt in (([3 << 20], C.MODE_FP32, C.F32), ([1 << 20] * 17, C.MODE_FP32, C.F32)):
        plan = _create(lib, _records(sizes, mode, fake), mode, gdt)
        try:
            lr, step = _scalars(fake)
            assert lib.adamw_step(plan, lr, step, 0.9, 0.999, 1e-8, None, None, None) == C.OK
            assert lib.probe_kind(0).decode() == "bulk", sizes
        finally:
            lib.adamw_plan_destroy(plan)
