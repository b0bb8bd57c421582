"""The bounded device-side waits of the bulk-staged step pipeline.

Every wait on an mbarrier in the step kernels gives up after a time limit,
records a fault bit that the host reads with adamw_plan_status, and leaves the
CUDA context usable.  The self-test makes a wait run out on purpose (a phase
that nothing completes) with a short limit and checks the reported status;
healthy plans report no fault after real steps.
"""

import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi as C

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    stream = torch.cuda.current_stream().cuda_stream
    status, ms = C.adamw_wait_selftest(50_000, stream)     # 50 ms limit
    assert status == C.ETIMEOUT
    assert 50.0 <= ms < 2000.0
    # the context is still usable: a plan runs a step and reports no fault
    n = 100_003
    p = torch.randn(n, device="cuda") * 0.02
    g = torch.randn(n, device="cuda") * 1e-3
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    opt = FusedAdamW([p], [g], [m], [v], [0.1])
    step = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        opt.step(torch.tensor([1e-3], device="cuda"), step)
    assert opt.status() == 0
    assert int(step.item()) == 3 and torch.isfinite(p).all()


@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
def test_healthy_plans_report_no_fault(mode):
    n = 3 * 4096 + 17
    if mode == "fp32":
        p, r = torch.randn(n, device="cuda"), None
    else:
        p = torch.randn(n, device="cuda").to(torch.bfloat16)
        r = torch.zeros(n, dtype=torch.int16, device="cuda")
    g = torch.randn(n, device="cuda").to(torch.bfloat16)
    m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    opt = FusedAdamW([p], [g], [m], [v], [0.0], mode=mode, param_rems=[r] if r is not None else None)
    step = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(5):
        opt.step(torch.tensor([1e-3], device="cuda"), step)
    assert opt.status() == 0 and int(step.item()) == 5
