"""adamw_step_noalloc against the plan-based step, through the C ABI.

Callers that cannot call cudaMalloc -- because a caching allocator already owns
the free device memory, because allocating inside their training or serving
loop is not allowed, or because their host application permits no allocation
outside its own pool -- cannot build a plan.  adamw_step_noalloc gives them the
same step on a static device array built into the library.  Its results must be
bit-identical to adamw_plan_create + adamw_step on the same inputs, call after
call: the array keeps whatever the previous call left in it, so the second call
checks that nothing stale leaks into the next step.  A skipped step (found_inf
set) must leave everything untouched on both paths, and the array's fault word
must read clear afterwards.

This file is collected last on purpose (a failure here leaves every other test
already run); it also passes on its own in a fresh process.
"""

import numpy as np
import pytest

from adamw_optimizer_step_tensor_gb300 import _capi as C
from oracle import adamw as OA

SIZES = [5000, 1, 8192, 16385, 0, 777, 40001]
B1, B2, EPS = OA.f32(0.9), OA.f32(0.999), OA.f32(1e-8)


def _torch_grad_dtype(gdt):
    import torch
    return {C.F32: torch.float32, C.F16: torch.float16, C.BF16: torch.bfloat16}[gdt]


def _pair(mode, gdt, rng):
    """Two identical copies (plan side, no-allocation side) of one tensor list."""
    import torch
    sides = ([], [])
    for i, n in enumerate(SIZES):
        m = rng.normal(0, 1e-3, n).astype(np.float32)
        v = (rng.normal(0, 1e-3, n) ** 2).astype(np.float32)
        if mode == C.MODE_FP32:
            p = rng.normal(0, 0.02, n).astype(np.float32)
            host = {"p": p, "rem": None}
        else:
            bits = rng.normal(0, 0.02, n).astype(np.float32).view(np.uint32)
            host = {"p": (bits >> 16).astype(np.uint16).view(np.int16),
                    "rem": rng.integers(0, 1 << 15, n).astype(np.int16)}
        for side in sides:
            t = {k: (torch.from_numpy(a.copy()).cuda() if a is not None else None)
                 for k, a in (("p", host["p"]), ("rem", host["rem"]), ("m", m), ("v", v))}
            t["g"] = torch.empty(n, dtype=_torch_grad_dtype(gdt), device="cuda")
            t["wd"] = 0.1 if i % 2 == 0 else 0.0
            side.append(t)
    return sides


def _records(side):
    def ptr(x):
        return None if x is None else x.data_ptr()
    return [C.adamw_tensor(ptr(t["p"]), ptr(t["rem"]), ptr(t["g"]), ptr(t["m"]), ptr(t["v"]),
                           None, None, t["p"].numel(), t["wd"]) for t in side]


def _same_bits(a, b):
    return np.array_equal(a.cpu().view(-1).numpy().view(np.uint8), b.cpu().view(-1).numpy().view(np.uint8))


def _snapshot(side):
    return [{k: t[k].clone() for k in ("p", "rem", "m", "v") if t[k] is not None} for t in side]


@pytest.mark.gpu
@pytest.mark.parametrize("gdt", [C.F32, C.F16, C.BF16], ids=["f32", "f16", "bf16"])
@pytest.mark.parametrize("mode", [C.MODE_FP32, C.MODE_BF16_REM], ids=["fp32", "bf16rem"])
def test_noalloc_step_equals_plan_step_on_two_calls(mode, gdt):
    import torch
    rng = np.random.default_rng(99)
    plan_side, free_side = _pair(mode, gdt, rng)
    plan = C.adamw_plan_create(_records(plan_side), mode, gdt)
    recs = _records(free_side)
    lr = torch.tensor([OA.f32(1e-2)], device="cuda")
    step_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    step_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the fp16 grads carry a loss scale, as they would under AMP
    scale = torch.tensor([1024.0 if gdt == C.F16 else 1.0], device="cuda")
    found = torch.zeros(1, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    try:
        for call in range(2):
            for a, b in zip(plan_side, free_side):
                g = rng.normal(0, 1e-3, a["g"].numel()) * (1024.0 if gdt == C.F16 else 1.0)
                a["g"].copy_(torch.from_numpy(g.astype(np.float32)).to(a["g"].dtype))
                b["g"].copy_(a["g"])
            C.adamw_step(plan, lr.data_ptr(), step_a.data_ptr(), B1, B2, EPS, scale.data_ptr(),
                         found.data_ptr(), stream)
            C.adamw_step_noalloc(recs, mode, gdt, lr.data_ptr(), step_b.data_ptr(), B1, B2, EPS,
                                 scale.data_ptr(), found.data_ptr(), stream)
            torch.cuda.synchronize()
            for i, (a, b) in enumerate(zip(plan_side, free_side)):
                for k in ("p", "rem", "m", "v"):
                    if a[k] is not None:
                        assert _same_bits(a[k], b[k]), f"call {call}: tensor {i} {k} differs"
            assert int(step_a.item()) == int(step_b.item()) == call + 1
        # a skipped step: found_inf set, nothing may change on either path
        before = _snapshot(free_side)
        found.fill_(1.0)
        C.adamw_step(plan, lr.data_ptr(), step_a.data_ptr(), B1, B2, EPS, scale.data_ptr(),
                     found.data_ptr(), stream)
        C.adamw_step_noalloc(recs, mode, gdt, lr.data_ptr(), step_b.data_ptr(), B1, B2, EPS,
                             scale.data_ptr(), found.data_ptr(), stream)
        torch.cuda.synchronize()
        for i, (a, b, s) in enumerate(zip(plan_side, free_side, before)):
            for k, t in s.items():
                assert _same_bits(a[k], t), f"skipped step changed plan-side tensor {i} {k}"
                assert _same_bits(b[k], t), f"skipped step changed tensor {i} {k}"
        assert int(step_a.item()) == int(step_b.item()) == 2
        assert C.adamw_step_noalloc_status() == 0
    finally:
        C.adamw_plan_destroy(plan)


def test_noalloc_rejects_what_the_static_array_cannot_hold():
    """Refused on the host, before any device access (runs without a GPU)."""
    rec = C.adamw_tensor(0x1000, None, 0x2000, 0x3000, 0x4000, None, None, 16, 0.0)
    with pytest.raises(C.AdamWError) as e:
        C.adamw_step_noalloc([rec] * 1025, C.MODE_FP32, C.F32, 0x100, 0x200, B1, B2, EPS,
                             None, None, None)
    assert e.value.status == C.EINVAL and "1024" in str(e.value)
    # one tensor needing more than 65536 chunks of at most 16384 elements
    big = C.adamw_tensor(0x1000, None, 0x2000, 0x3000, 0x4000, None, None, 65536 * 16384 + 1, 0.0)
    with pytest.raises(C.AdamWError) as e:
        C.adamw_step_noalloc([big], C.MODE_FP32, C.F32, 0x100, 0x200, B1, B2, EPS, None, None, None)
    assert e.value.status == C.EINVAL and "65536" in str(e.value)
    with pytest.raises(C.AdamWError) as e:
        C.adamw_step_noalloc([rec], C.MODE_Q8, C.F32, 0x100, 0x200, B1, B2, EPS, None, None, None)
    assert e.value.status == C.EUNSUPPORTED
    with pytest.raises(C.AdamWError) as e:
        C.adamw_step_noalloc([rec], 7, C.F32, 0x100, 0x200, B1, B2, EPS, None, None, None)
    assert e.value.status == C.EDTYPE
    # the same eps rule as adamw_step
    with pytest.raises(C.AdamWError) as e:
        C.adamw_step_noalloc([rec], C.MODE_FP32, C.F32, 0x100, 0x200, B1, B2, float("inf"),
                             None, None, None)
    assert e.value.status == C.EINVAL and "eps" in str(e.value)
