#!/usr/bin/env python3
"""Throughput of the fused AdamW step on GB300 (params/s and achieved HBM GB/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3_8b|gpt2_small|single|amp|amp_fused|q8|q4|bf16rem|
                                ademamix_gpt2|lion_gpt2|momentum_gpt2|rmsprop_gpt2|adagrad_gpt2|
                                adam_mini_llama3]

One "step" is one optimizer update of every tensor of the workload (one launch
of the library's step kernel; plus the non-finite check in the AMP workload).
The default workload is the largest one that fits one GPU: the Llama-3-8B
parameter list (291 tensors, 8,030,261,248 elements) as bf16 params with int16
remainders, bf16 grads, fp32 m and v, lr from a device tensor (209 GB moved per
step, far larger than L2).  The GPT-2-small fp32 list, the single-tensor and
AMP cases, the 8-bit and 4-bit states and the other update rules are the
other workloads; the L2-resident single-tensor ones flush L2 between timed
launches.  Inputs are synthetic and seeded (``synth``), resident in HBM before
timing.  Under torchrun every rank runs its own copy of the workload on its own
GPU (weak scaling; the update is element-wise and needs no exchange).

The end-to-end arm (``e2e``) runs the same step through the C ABI with the
grads copied in from pinned host memory and the updated params copied back,
every step, inside the timed region.  ``cpu_baseline`` times the CPU oracle on
every host core (one process per core).  ``--impl reference`` times the CPU
oracle alone on a bounded sample of the same workload, on every host core.
One JSON line is printed by rank 0.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "optimizer-step params/sec and achieved HBM GB/s (% of GB300 peak)"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0        # the GB300's nominal HBM3e bandwidth, reported beside the measured peak
L2_FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b",
                    choices=["gpt2_small", "single", "amp", "amp_fused", "q8", "llama3_8b", "bf16rem",
                             "ademamix_gpt2", "lion_gpt2", "momentum_gpt2", "rmsprop_gpt2",
                             "adagrad_gpt2", "q4", "adam_mini_llama3"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-l2-flush", action="store_true",
                    help="single/amp workloads: keep L2 between timed launches (L2-resident rate)")
    ap.add_argument("--numel", type=int, default=0,
                    help="element count override for the single/amp/q8 workloads (profiling)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


# The source files that make up the dominant kernel of each workload; a
# committed ncu summary counts only while their hash matches.
SMALL_SOURCES = ("small_kernels.cu", "step_common.cuh", "internal.h", "async_copy.cuh")
KERNEL_SOURCES = {
    "q8": ("step_kernels.cu", "step_common.cuh", "internal.h", "lane_tables.cuh"),
    "q4": ("q4_kernels.cu", "step_common.cuh", "internal.h"),
    "single": SMALL_SOURCES, "amp": SMALL_SOURCES, "amp_fused": SMALL_SOURCES,
}
BULK_SOURCES = ("bulk_kernels.cu", "step_common.cuh", "internal.h", "async_copy.cuh")


def kernel_source_sha(workload: str = "gpt2_small") -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "adamw_optimizer_step_tensor_gb300", "csrc")
    for name in KERNEL_SOURCES.get(workload, BULK_SOURCES):
        with open(os.path.join(d, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_figure(workload: str, key: str):
    """A figure from the committed ncu summary of the workload's kernel, if the
    summary still matches the source."""
    path = os.path.join(ROOT, "profiles", f"step_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    val = re.search(key + r":\s*([0-9.eE+]+)", txt)
    if not sha or not val or sha.group(1) != kernel_source_sha(workload):
        return None
    return float(val.group(1))


def ncu_traffic(workload: str):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)."""
    return ncu_figure(workload, "dram_bytes_per_launch")


def issue_roofline(workload: str, elems_per_s: float, sm_mhz, sms: int | None = None):
    """The second roofline of the step kernels, instruction issue: ncu's warp
    instructions per element times the element rate, against one warp
    instruction per scheduler per cycle (4 schedulers per SM) at the SM clock
    sampled during the timed region (the device's SM count unless given)."""
    wpe = ncu_figure(workload, "warp_instructions_per_element")
    if wpe is None:
        return None
    if sms is None:
        import torch
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = sm_mhz or 2070.0
    peak = sms * 4 * mhz * 1e6
    achieved = wpe * elems_per_s
    return {"bound": "issue", "warp_inst_per_element": wpe, "achieved": achieved, "peak": peak,
            "unit": "warp-inst/s", "frac": achieved / peak,
            "peak_source": f"{sms} SMs x 4 schedulers x {mhz:.0f} MHz (sampled SM clock)"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t_begin: float, t_end: float):
        import datetime
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        sel = [r for r in rows if t_begin <= r[0] <= t_end]
        note = None
        if len(sel) < 3:
            sel = rows
            note = (f"timed region {(t_end - t_begin) * 1e3:.0f} ms holds fewer than 3 of the 200 ms "
                    "samples; median over the whole run (warm-up and timed steps)")
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i in range(4) if r[3][i].lower() == "active"})
        out = {"sm_mhz": statistics.median(r[1] for r in sel),
               "sm_max_mhz": max(r[2] for r in sel), "reasons": reasons, "samples": len(sel)}
        if note:
            out["note"] = note
        return out


def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())



# ----------------------------------------------------------------------------- CPU samples
def cpu_sample_fp32(n, amp=False, lr=1e-3, wd=0.1):
    """One float64-oracle step over n elements per call (fp32-state workloads)."""
    import numpy as np
    from oracle import adamw as OA
    rng = np.random.default_rng(0)
    scale = 65536.0 if amp else None
    g = rng.normal(0, 1e-3, n) * (scale or 1.0)
    x = OA.Tensor(p=rng.normal(0, 0.02, n), g=g, m=np.zeros(n), v=np.zeros(n), wd=wd)
    state = {"t": 0}

    def run():
        state["t"] += 1
        OA.step_fp64([x], lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, t=state["t"], grad_scale=scale)
    return run, f"{n} elements per step, float64 oracle (oracle.adamw.step_fp64)"


def cpu_sample_fp32_strict(n, amp=False, lr=1e-3, wd=0.1):
    """One strict-fp32-oracle step over n elements per call (fp32-state workloads)."""
    import numpy as np
    from oracle import adamw as OA
    rng = np.random.default_rng(0)
    scale = 65536.0 if amp else None
    g = (rng.normal(0, 1e-3, n) * (scale or 1.0)).astype(np.float32)
    x = OA.Tensor(p=rng.normal(0, 0.02, n).astype(np.float32), g=g,
                  m=np.zeros(n, np.float32), v=np.zeros(n, np.float32), wd=OA.f32(wd))
    state = {"t": 0}

    def run():
        state["t"] += 1
        OA.step_f32([x], lr=OA.f32(lr), beta1=OA.f32(0.9), beta2=OA.f32(0.999), eps=OA.f32(1e-8),
                    t=state["t"], grad_scale=scale)
    return run, f"{n} elements per step, strict-fp32 oracle (oracle.adamw.step_f32)"


def cpu_sample_q8(n):
    import numpy as np
    from oracle import q8 as OQ
    n = max(256, n // 256 * 256)
    rng = np.random.default_rng(0)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    cm, cv = np.zeros(n, np.uint8), np.zeros(n, np.uint8)
    am, av = np.zeros(n // 256, np.float32), np.zeros(n // 256, np.float32)
    maps = OQ.Maps()
    state = {"t": 0}

    def run():
        state["t"] += 1
        OQ.step_f32(p, g, cm, cv, am, av, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01,
                    t=state["t"], maps=maps)
    return run, f"{n} elements per step, strict-fp32 8-bit-state oracle (oracle.q8.step_f32)"


def cpu_sample_bf16rem(n):
    import numpy as np
    from oracle import adamw as OA, remainder as OR
    rng = np.random.default_rng(0)
    hi = (rng.normal(0, 0.02, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    rem = rng.integers(0, 1 << 15, n).astype(np.int16)
    g = rng.normal(0, 1e-4, n).astype(np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    state = {"t": 0, "hi": hi, "rem": rem}

    def run():
        state["t"] += 1
        x = OA.Tensor(p=OR.join(state["hi"], state["rem"]), g=g, m=m, v=v, wd=0.1)
        OA.step_f32([x], lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, t=state["t"])
        state["hi"], state["rem"] = OR.split(x.p)
    return run, f"{n} elements per step, strict-fp32 oracle with remainder join/split"


def cpu_sample_q4(n):
    import numpy as np
    from oracle import q4 as O4
    n = max(128, n // 128 * 128)
    rng = np.random.default_rng(0)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    pm, pv = np.zeros(n // 2, np.uint8), np.zeros(n // 2, np.uint8)
    am, av = np.zeros(n // 128, np.float32), np.zeros(n // 128, np.float32)
    maps = O4.Maps4()
    state = {"t": 0}

    def run():
        state["t"] += 1
        O4.step_f32(p, g, pm, pv, am, av, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01,
                    t=state["t"], maps=maps)
    return run, f"{n} elements per step, strict-fp32 4-bit oracle (oracle.q4.step_f32)"


def cpu_sample_mini(n):
    import numpy as np
    from oracle import mini as OM
    block = 524288
    n = max(block, n // block * block)
    rng = np.random.default_rng(0)
    x = OM.Tensor(p=rng.normal(0, 0.02, n), g=rng.normal(0, 1e-4, n), m=np.zeros(n),
                  v=np.zeros(n // block), wd=0.1, block=block)
    state = {"t": 0}

    def run():
        state["t"] += 1
        OM.step_fp64([x], lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, t=state["t"])
    return run, f"{n} elements per step in heads of {block}, float64 Adam-mini oracle (oracle.mini.step_fp64)"


def cpu_sample_ademamix(n):
    import numpy as np
    from oracle import ademamix as OX
    rng = np.random.default_rng(0)
    x = OX.Tensor(p=rng.normal(0, 0.02, n), g=rng.normal(0, 1e-3, n), m1=np.zeros(n), m2=np.zeros(n),
                  v=np.zeros(n), wd=0.1)
    state = {"t": 0}

    def run():
        state["t"] += 1
        OX.step_fp64([x], lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0, eps=1e-8,
                     t=state["t"])
    return run, f"{n} elements per step, float64 AdEMAMix oracle (oracle.ademamix.step_fp64)"


def cpu_sample_lion(n):
    import numpy as np
    from oracle import lion as OL
    rng = np.random.default_rng(0)
    x = OL.Tensor(p=rng.normal(0, 0.02, n), g=rng.normal(0, 1e-3, n), m=np.zeros(n), wd=0.1)

    def run():
        OL.step_fp64([x], lr=1e-4, beta1=0.9, beta2=0.99)
    return run, f"{n} elements per step, float64 Lion oracle (oracle.lion.step_fp64)"


def cpu_sample_coupled(n, rule):
    import numpy as np
    from oracle import coupled as OC
    rng = np.random.default_rng(0)
    x = OC.Tensor(p=rng.normal(0, 0.02, n), g=rng.normal(0, 1e-3, n), s=np.zeros(n), wd=0.1)

    def run():
        OC.step_fp64([x], rule=rule, lr=1e-3, beta=0.9, eps=1e-8)
    return run, f"{n} elements per step, float64 {rule} oracle (oracle.coupled.step_fp64)"


def cpu_sample_bf16rem_fp64(n):
    """The float64 definition on the bf16+remainder layout: join to the float32
    master, one float64 step, round to float32 and split again."""
    import numpy as np
    from oracle import adamw as OA, remainder as OR
    rng = np.random.default_rng(0)
    hi = (rng.normal(0, 0.02, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    rem = rng.integers(0, 1 << 15, n).astype(np.int16)
    g = rng.normal(0, 1e-4, n)
    m, v = np.zeros(n), np.zeros(n)
    state = {"t": 0, "hi": hi, "rem": rem}

    def run():
        state["t"] += 1
        x = OA.Tensor(p=OR.join(state["hi"], state["rem"]).astype(np.float64), g=g, m=m, v=v, wd=0.1)
        OA.step_fp64([x], lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, t=state["t"])
        state["hi"], state["rem"] = OR.split(x.p.astype(np.float32))
    return run, (f"{n} elements per step, float64 definition (oracle.adamw.step_fp64) on the "
                 "joined master, rounded to float32 and split")


# A second oracle timed beside the first: strict fp32 beside the float64
# definition (fp32-state AdamW workloads), the float64 definition beside the
# strict-fp32 remainder oracle (bf16+remainder workloads).
CPU_SAMPLES_SECOND = {
    "gpt2_small": ("strict_fp32", lambda n: cpu_sample_fp32_strict(n)),
    "single": ("strict_fp32", lambda n: cpu_sample_fp32_strict(n, lr=0.1)),
    "amp": ("strict_fp32", lambda n: cpu_sample_fp32_strict(n, amp=True, lr=0.1)),
    "amp_fused": ("strict_fp32", lambda n: cpu_sample_fp32_strict(n, amp=True, lr=0.1)),
    "llama3_8b": ("fp64", cpu_sample_bf16rem_fp64),
    "bf16rem": ("fp64", cpu_sample_bf16rem_fp64),
}

# The arithmetic type of each workload's first CPU oracle (the reference arm).
REFERENCE_DTYPE = {"q8": "f32", "q4": "f32", "llama3_8b": "f32", "bf16rem": "f32"}

CPU_SAMPLES = {
    "gpt2_small": lambda n: cpu_sample_fp32(n),
    "single": lambda n: cpu_sample_fp32(n, lr=0.1),
    "amp": lambda n: cpu_sample_fp32(n, amp=True, lr=0.1),
    "amp_fused": lambda n: cpu_sample_fp32(n, amp=True, lr=0.1),
    "q8": cpu_sample_q8,
    "llama3_8b": cpu_sample_bf16rem,
    "bf16rem": cpu_sample_bf16rem,
    "ademamix_gpt2": lambda n: cpu_sample_ademamix(n),
    "lion_gpt2": lambda n: cpu_sample_lion(n),
    "momentum_gpt2": lambda n: cpu_sample_coupled(n, "momentum"),
    "rmsprop_gpt2": lambda n: cpu_sample_coupled(n, "rmsprop"),
    "adagrad_gpt2": lambda n: cpu_sample_coupled(n, "adagrad"),
    "q4": lambda n: cpu_sample_q4(n),
    "adam_mini_llama3": lambda n: cpu_sample_mini(n),
}

# ----------------------------------------------------------------------------- workloads
def _flat_views(specs, dtype, device, fill=None, align=64):
    """One contiguous buffer holding every tensor, each starting 256-byte aligned."""
    import torch
    offs, o = [], 0
    for s in specs:
        offs.append(o)
        o += (s.numel + align - 1) // align * align
    buf = torch.zeros(o, dtype=dtype, device=device)
    views = [buf[a:a + s.numel] for a, s in zip(offs, specs)]
    return buf, views


class Workload:
    name = ""
    bytes_per_param = 0.0
    n_params = 0
    launches_per_step = 1
    flush_l2 = False
    dtype = "f32"

    def step(self, i):  # one optimizer step on the current stream
        raise NotImplementedError

    def e2e_step(self, i):
        raise NotImplementedError



class PipelinedE2E:
    """The host-offload arm of a workload: every step its grads arrive from
    pinned host memory and its updated params go back.  The elements are cut
    into groups with one plan (and step counter) each, so that the
    host-to-device copy of one group, the step of the previous one and the
    device-to-host copy of the one before overlap on three streams.

    Without a ring the host holds a full pinned copy of every buffer.  With
    ``ring`` = R the host holds R group-sized slots per buffer and group k
    goes through slot k mod R (its grads come from that slot, its results
    land in it): a bounded host footprint for lists whose buffers do not fit
    in pinned host memory.  Each copy of a group is one contiguous range of a
    flat device buffer."""

    def _pipeline(self, ins, outs, groups, ring=None):
        """ins / outs: flat device buffers copied in / out every step;
        groups: (lo, hi, plan) over their element ranges."""
        import torch
        self._ins, self._outs = list(ins), list(outs)
        self._groups = [(lo, hi, opt, torch.zeros(1, dtype=torch.int32, device="cuda"))
                        for lo, hi, opt in groups]
        self._ring = ring
        if ring is None:
            self._host_in = [torch.empty_like(b, device="cpu").pin_memory() for b in self._ins]
            for h, b in zip(self._host_in, self._ins):
                h.copy_(b)
            self._host_out = [torch.empty_like(b, device="cpu").pin_memory() for b in self._outs]
        else:
            width = max(hi - lo for lo, hi, _ in groups)
            self._host_in = [torch.empty((ring, width), dtype=b.dtype).pin_memory() for b in self._ins]
            self._host_out = [torch.empty((ring, width), dtype=b.dtype).pin_memory() for b in self._outs]
            for j, (lo, hi, _) in enumerate(groups[:ring]):      # slot j starts as group j's grads
                for h, b in zip(self._host_in, self._ins):
                    h[j, :hi - lo].copy_(b[lo:hi])
        self._s = [torch.cuda.Stream() for _ in range(3)]          # in, step, out
        n = len(self._groups)
        self._ev = [[torch.cuda.Event() for _ in range(n)] for _ in range(3)]
        span = sum(hi - lo for lo, hi, _ in groups)
        return (sum(span * b.element_size() for b in self._ins),
                sum(span * b.element_size() for b in self._outs))

    def _host_range(self, h, k, lo, hi):
        return h[lo:hi] if self._ring is None else h[k % self._ring, :hi - lo]

    def e2e_begin(self, stream):
        for s in self._s:
            s.wait_stream(stream)

    def e2e_end(self, stream):
        for s in self._s:
            stream.wait_stream(s)

    def e2e_step(self, i):
        import torch
        s_in, s_cmp, s_out = self._s
        ev_in, ev_cmp, ev_out = self._ev
        for k, (lo, hi, opt, step_dev) in enumerate(self._groups):
            s_in.wait_event(ev_cmp[k])            # the previous step has consumed these grads
            with torch.cuda.stream(s_in):
                for h, b in zip(self._host_in, self._ins):
                    b[lo:hi].copy_(self._host_range(h, k, lo, hi), non_blocking=True)
            ev_in[k].record(s_in)
            s_cmp.wait_event(ev_in[k])
            s_cmp.wait_event(ev_out[k])           # the previous copy-out has read these params
            self._group_step(opt, i, step_dev, s_cmp.cuda_stream)
            ev_cmp[k].record(s_cmp)
            s_out.wait_event(ev_cmp[k])
            with torch.cuda.stream(s_out):
                for h, b in zip(self._host_out, self._outs):
                    self._host_range(h, k, lo, hi).copy_(b[lo:hi], non_blocking=True)
            ev_out[k].record(s_out)


class Gpt2Small(PipelinedE2E, Workload):
    name = "gpt2_small_fp32_cosine_lr"
    bytes_per_param = 28.0
    e2e_what = ("pinned-host grads -> device, adamw_step, updated params -> pinned host; the list "
                "in 8 groups (one plan each) so copies in, steps and copies out overlap on 3 streams")

    def __init__(self, seed=0):
        import torch
        import synth
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi
        dev = torch.device("cuda")
        self.C = _capi
        self.specs = synth.gpt2_small()
        self.n_params = synth.total_numel(self.specs)
        self.p_buf, ps = _flat_views(self.specs, torch.float32, dev)
        self.g_buf, gs = _flat_views(self.specs, torch.float32, dev)
        self.g2_buf, gs2 = _flat_views(self.specs, torch.float32, dev)
        self.m_buf, ms = _flat_views(self.specs, torch.float32, dev)
        self.v_buf, vs = _flat_views(self.specs, torch.float32, dev)
        for i, (p, g, g2) in enumerate(zip(ps, gs, gs2)):
            p.copy_(synth.normal(p.numel(), 0.02, seed + i, dev))
            g.copy_(synth.normal(g.numel(), 1e-3, synth.grad_seed(seed, 0, i), dev))
            g2.copy_(synth.normal(g2.numel(), 1e-3, synth.grad_seed(seed, 1, i), dev))
        self.ps, self.gs, self.gs2, self.ms, self.vs = ps, gs, gs2, ms, vs
        # two grad sets, one plan each, alternating step by step: with one
        # fixed set, coupled weight decay drives p to -g/wd and the state of
        # RMSprop towards subnormal values (slow division and square root)
        self.opts = [FusedAdamW(ps, g, ms, vs, [s.wd for s in self.specs]) for g in (gs, gs2)]
        self.lr_table = torch.tensor([synth.cosine_lr(s) for s in range(100)], dtype=torch.float32,
                                     device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        self.lr_ptrs = [self.lr_table.data_ptr() + 4 * s for s in range(100)]
        self.stream = torch.cuda.current_stream().cuda_stream
        self.config = Gpt2Small.describe()
        self._host = None

    @classmethod
    def describe(cls, seed=0):
        import synth
        specs = synth.gpt2_small()
        return {"workload": "gpt2_small fp32 param list, cosine lr from a device table",
                "tensors": len(specs), "numel": synth.total_numel(specs),
                "bytes_per_param": Gpt2Small.bytes_per_param,
                "grad_dtype": "f32", "state_dtype": "f32",
                "grads": "two seeded N(0,1e-3) sets, alternating step by step",
                "l2": "no flush: 3.48 GB moved per step, larger than the 126 MB L2",
                "lr_schedule": "cosine 1e-3 -> 1e-4 over 100 steps, lr_dev points into it"}

    def step(self, i):
        self.C.adamw_step(self.opts[i % 2].plan, self.lr_ptrs[i % 100], self.step_dev.data_ptr(),
                          0.9, 0.999, 1e-8, None, None, self.stream)

    def step_grads(self, i):
        """The grad tensors that step i reads (the two sets alternate)."""
        return self.gs if i % 2 == 0 else self.gs2

    def status(self) -> int:
        """Device-side fault bits of every plan, or-ed."""
        out = 0
        for o in self.opts:
            out |= o.status()
        return out

    def e2e_setup(self, groups=8):
        """The list in `groups` contiguous runs of tensors of about equal element
        counts (PipelinedE2E)."""
        base = self.p_buf.data_ptr()
        offs = [(p.data_ptr() - base) // 4 for p in self.ps]
        target = self.n_params / groups
        runs, start, acc = [], 0, 0
        for k, p in enumerate(self.ps):
            acc += p.numel()
            if acc >= target * (len(runs) + 1) or k == len(self.ps) - 1:
                idx = list(range(start, k + 1))
                runs.append((offs[start], offs[k] + self.ps[k].numel(), self._group_plan(idx)))
                start = k + 1
        return self._pipeline([self.g_buf], [self.p_buf], runs)

    def _group_plan(self, idx):
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW
        return FusedAdamW([self.ps[j] for j in idx], [self.gs[j] for j in idx],
                          [self.ms[j] for j in idx], [self.vs[j] for j in idx],
                          [self.specs[j].wd for j in idx])

    def _group_step(self, opt, i, step_dev, stream):
        self.C.adamw_step(opt.plan, self.lr_ptrs[i % 100], step_dev.data_ptr(), 0.9, 0.999, 1e-8,
                          None, None, stream)


class AdemamixGpt2(Gpt2Small):
    """The GPT-2-small list stepped with AdEMAMix (a third fp32 state: 36 B/element)."""
    name = "ademamix_gpt2_small_fp32"
    bytes_per_param = 36.0

    def __init__(self, seed=0):
        import torch
        super().__init__(seed)
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW
        self.m2_buf, m2s = _flat_views(self.specs, torch.float32, torch.device("cuda"))
        self.m2s = m2s
        self.opts = [FusedAdamW(self.ps, g, self.ms, self.vs, [s.wd for s in self.specs],
                                exp_avg_slows=m2s) for g in (self.gs, self.gs2)]
        self.config = AdemamixGpt2.describe()
        self.e2e_what = self.e2e_what.replace("adamw_step", "adamw_ademamix_step")

    @classmethod
    def describe(cls, seed=0):
        return dict(Gpt2Small.describe(), workload="gpt2_small fp32 param list, AdEMAMix (m1, m2, v), "
                    "cosine lr from a device table", bytes_per_param=AdemamixGpt2.bytes_per_param,
                    l2="no flush: 4.48 GB moved per step, larger than the 126 MB L2")

    def step(self, i):
        self.C.adamw_ademamix_step(self.opts[i % 2].plan, self.lr_ptrs[i % 100], self.step_dev.data_ptr(),
                                   0.9, 0.999, 0.9999, 5.0, 1e-8, None, None, self.stream)

    def _group_plan(self, idx):
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW
        return FusedAdamW([self.ps[j] for j in idx], [self.gs[j] for j in idx],
                          [self.ms[j] for j in idx], [self.vs[j] for j in idx],
                          [self.specs[j].wd for j in idx], exp_avg_slows=[self.m2s[j] for j in idx])

    def _group_step(self, opt, i, step_dev, stream):
        self.C.adamw_ademamix_step(opt.plan, self.lr_ptrs[i % 100], step_dev.data_ptr(), 0.9, 0.999,
                                   0.9999, 5.0, 1e-8, None, None, stream)


class LionGpt2(Gpt2Small):
    """The GPT-2-small list stepped with Lion (one fp32 state, no v: 20 B/element)."""
    name = "lion_gpt2_small_fp32"
    bytes_per_param = 20.0

    def __init__(self, seed=0):
        super().__init__(seed)
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW
        self.opts = [FusedAdamW(self.ps, g, self.ms, None, [s.wd for s in self.specs])
                     for g in (self.gs, self.gs2)]
        self.vs = self.v_buf = None
        self.config = LionGpt2.describe()
        self.e2e_what = self.e2e_what.replace("adamw_step", "adamw_lion_step")

    @classmethod
    def describe(cls, seed=0):
        return dict(Gpt2Small.describe(), workload="gpt2_small fp32 param list, Lion (m only), "
                    "cosine lr from a device table", bytes_per_param=LionGpt2.bytes_per_param,
                    l2="no flush: 2.49 GB moved per step, larger than the 126 MB L2")

    def step(self, i):
        self.C.adamw_lion_step(self.opts[i % 2].plan, self.lr_ptrs[i % 100], self.step_dev.data_ptr(),
                               0.9, 0.99, None, None, self.stream)

    def _group_plan(self, idx):
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW
        return FusedAdamW([self.ps[j] for j in idx], [self.gs[j] for j in idx],
                          [self.ms[j] for j in idx], None, [self.specs[j].wd for j in idx])

    def _group_step(self, opt, i, step_dev, stream):
        self.C.adamw_lion_step(opt.plan, self.lr_ptrs[i % 100], step_dev.data_ptr(), 0.9, 0.99,
                               None, None, stream)


class CoupledGpt2(LionGpt2):
    """The GPT-2-small list stepped with momentum SGD, RMSprop or Adagrad (coupled
    L2; one fp32 state, no v: 20 B/element)."""
    bytes_per_param = 20.0

    def __init__(self, rule, seed=0):
        super().__init__(seed)
        self.rule = rule
        self.rule_id = self.C.RULES[rule]
        self.name = f"{rule}_gpt2_small_fp32"
        self.config = CoupledGpt2.describe(rule)
        self.e2e_what = self.e2e_what.replace("adamw_lion_step", "adamw_coupled_step")

    @classmethod
    def describe(cls, rule, seed=0):
        return dict(LionGpt2.describe(), workload=f"gpt2_small fp32 param list, {rule} with coupled "
                    "L2 (one state), cosine lr from a device table")

    def step(self, i):
        self.C.adamw_coupled_step(self.opts[i % 2].plan, self.rule_id, self.lr_ptrs[i % 100],
                                  self.step_dev.data_ptr(), 0.9, 1e-8, None, None, self.stream)

    def _group_step(self, opt, i, step_dev, stream):
        self.C.adamw_coupled_step(opt.plan, self.rule_id, self.lr_ptrs[i % 100], step_dev.data_ptr(),
                                  0.9, 1e-8, None, None, stream)


class Single(Workload):
    name = "single_fp32_1M_l2flush"
    bytes_per_param = 28.0
    flush_l2 = True

    def __init__(self, amp=False, seed=1, numel=0, fused=False):
        import torch
        import synth
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi
        dev = torch.device("cuda")
        self.C = _capi
        self.amp = amp
        n = self.n_params = numel or (1 << 20)
        self.p = synth.normal(n, 0.02, seed, dev)
        gd = torch.float16 if amp else torch.float32
        self.g = (synth.normal(n, 1e-3, seed + 1, dev) * (65536.0 if amp else 1.0)).to(gd)
        self.m = torch.zeros(n, device=dev)
        self.v = torch.zeros(n, device=dev)
        self.opt = FusedAdamW([self.p], [self.g], [self.m], [self.v], [0.1])
        self.lr = torch.tensor([0.1], dtype=torch.float32, device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        self.scale = torch.tensor([65536.0], device=dev)
        self.found = torch.zeros(1, device=dev)
        self.stream = torch.cuda.current_stream().cuda_stream
        self.fused = fused
        # adamw_step_amp runs the check and the step as two launches above 6 Mi elements
        self.launches_per_step = 2 if amp and (not fused or n > (6 << 20)) else 1
        if amp:
            self.name = "amp_fp16_grads_1M_l2flush"
            self.bytes_per_param = 28.0
            self.inject = synth.amp_injection(10 ** 6, n, seed=3)
        self.config = Single.describe(amp=amp, numel=numel, fused=fused)

    @classmethod
    def describe(cls, amp=False, seed=1, numel=0, fused=False):
        return {"workload": ("AMP fp16 grads x65536, unscale + found_inf skip, 1 tensor, "
                             + ("check and step in one launch (adamw_step_amp)" if fused
                                else "check and step as two launches")
                             if amp else "single fp32 tensor"),
                "tensors": 1, "numel": numel or (1 << 20), "bytes_per_param": 28.0,
                "l2": f"L2 flushed ({L2_FLUSH_BYTES >> 20} MB write) before every timed launch; "
                      "launch times summed"}

    def step(self, i):
        if self.amp and self.fused:
            self.C.adamw_step_amp(self.opt.plan, self.lr.data_ptr(), self.step_dev.data_ptr(), 0.9,
                                  0.999, 1e-8, self.scale.data_ptr(), self.found.data_ptr(),
                                  self.stream)
        elif self.amp:
            self.C.adamw_check_nonfinite(self.opt.plan, self.found.data_ptr(), self.stream)
            self.C.adamw_step(self.opt.plan, self.lr.data_ptr(), self.step_dev.data_ptr(), 0.9, 0.999,
                              1e-8, self.scale.data_ptr(), self.found.data_ptr(), self.stream)
        else:
            self.C.adamw_step(self.opt.plan, self.lr.data_ptr(), self.step_dev.data_ptr(), 0.9, 0.999,
                              1e-8, None, None, self.stream)

    def e2e_setup(self):
        import torch
        self._host_g = torch.empty_like(self.g, device="cpu").pin_memory()
        self._host_g.copy_(self.g)
        self._host_p = torch.empty_like(self.p, device="cpu").pin_memory()
        return self._host_g.numel() * self._host_g.element_size(), self._host_p.numel() * 4

    def e2e_step(self, i):
        self.g.copy_(self._host_g, non_blocking=True)
        self.step(i)
        self._host_p.copy_(self.p, non_blocking=True)



class Q8(PipelinedE2E, Workload):
    name = "q8_blockwise_1G"
    bytes_per_param = 14.0625
    mode, block, codes_per_byte = "q8", 256, 1
    e2e_what = ("pinned-host grads -> device, adamw_step, updated params -> pinned host; the "
                "tensor in 8 slices (one plan each) so copies in, steps and copies out overlap "
                "on 3 streams")

    def __init__(self, seed=4, numel=0):
        import torch
        import synth
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi
        dev = torch.device("cuda")
        self.C = _capi
        n = self.n_params = numel or (1 << 30)
        self.p = synth.normal(n, 0.02, seed, dev)
        self.g = synth.normal(n, 1e-3, seed + 1, dev, dtype=torch.bfloat16)
        self.cm = torch.zeros(n, dtype=torch.uint8, device=dev)
        self.cv = torch.zeros(n, dtype=torch.uint8, device=dev)
        nb = (n + 255) // 256
        self.am = torch.zeros(nb, device=dev)
        self.av = torch.zeros(nb, device=dev)
        self.opt = FusedAdamW([self.p], [self.g], [self.cm], [self.cv], [0.01], mode="q8",
                              absmax_m=[self.am], absmax_v=[self.av])
        self.lr = torch.tensor([1e-3], dtype=torch.float32, device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream().cuda_stream
        self.dtype = "f32 (u8 states)"
        self.config = Q8.describe(numel=numel)

    @classmethod
    def describe(cls, seed=4, numel=0):
        return {"workload": "8-bit blockwise m,v; one flat fp32 param of 2^30, bf16 grads",
                "tensors": 1, "numel": numel or (1 << 30), "bytes_per_param": Q8.bytes_per_param,
                "l2": "no flush: 15.1 GB moved per step"}

    def step(self, i):
        self.C.adamw_step(self.opt.plan, self.lr.data_ptr(), self.step_dev.data_ptr(), 0.9, 0.999,
                          1e-8, None, None, self.stream)

    def e2e_setup(self, groups=8):
        """The tensor in `groups` slices of whole blocks, one plan each (PipelinedE2E)."""
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW
        n, b, cpb = self.n_params, self.block, self.codes_per_byte
        size = -(-n // groups // b) * b
        runs = []
        for lo in range(0, n, size):
            hi = min(n, lo + size)
            c0, c1 = lo // cpb, -(-hi // cpb)
            a0, a1 = lo // b, -(-hi // b)
            opt = FusedAdamW([self.p[lo:hi]], [self.g[lo:hi]], [self.cm[c0:c1]], [self.cv[c0:c1]],
                             [0.01], mode=self.mode, absmax_m=[self.am[a0:a1]],
                             absmax_v=[self.av[a0:a1]])
            runs.append((lo, hi, opt))
        return self._pipeline([self.g], [self.p], runs)

    def _group_step(self, opt, i, step_dev, stream):
        self.C.adamw_step(opt.plan, self.lr.data_ptr(), step_dev.data_ptr(), 0.9, 0.999, 1e-8,
                          None, None, stream)



class Q4(Q8):
    """The q8 workload with 4-bit packed codes and 128-element blocks."""
    name = "q4_blockwise_1G"
    bytes_per_param = 12.125      # p 4+4, g 2, codes 0.5+0.5 each way, absmax 8/128 each way
    mode, block, codes_per_byte = "q4", 128, 2

    def __init__(self, seed=4, numel=0):
        import torch
        import synth
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi
        dev = torch.device("cuda")
        self.C = _capi
        n = self.n_params = numel or (1 << 30)
        self.p = synth.normal(n, 0.02, seed, dev)
        self.g = synth.normal(n, 1e-3, seed + 1, dev, dtype=torch.bfloat16)
        self.cm = torch.zeros((n + 1) // 2, dtype=torch.uint8, device=dev)
        self.cv = torch.zeros((n + 1) // 2, dtype=torch.uint8, device=dev)
        nb = (n + 127) // 128
        self.am = torch.zeros(nb, device=dev)
        self.av = torch.zeros(nb, device=dev)
        self.opt = FusedAdamW([self.p], [self.g], [self.cm], [self.cv], [0.01], mode="q4",
                              absmax_m=[self.am], absmax_v=[self.av])
        self.lr = torch.tensor([1e-3], dtype=torch.float32, device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream().cuda_stream
        self.dtype = "f32 (4-bit states)"
        self.config = Q4.describe(numel=numel)

    @classmethod
    def describe(cls, seed=4, numel=0):
        return {"workload": "4-bit blockwise m,v (128-element blocks); one flat fp32 param "
                            "of 2^30, bf16 grads",
                "tensors": 1, "numel": numel or (1 << 30), "bytes_per_param": Q4.bytes_per_param,
                "l2": "no flush: 13.0 GB moved per step"}


class Llama3(PipelinedE2E, Workload):
    name = "llama3_8b_bf16_rem"
    bytes_per_param = 26.0
    e2e_steps = 8
    e2e_what = ("pinned-host bf16 grads -> device, adamw_step, updated bf16 params and int16 "
                "remainders -> pinned host; the flat list in 2^27-element groups (one plan "
                "each) through a 3-slot pinned host ring, so copies in, steps and copies out "
                "overlap on 3 streams")

    def __init__(self, seed=5):
        import torch
        import synth
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi
        dev = torch.device("cuda")
        self.C = _capi
        self.specs = synth.llama3_8b()
        self.n_params = synth.total_numel(self.specs)
        self.h_buf, hs = _flat_views(self.specs, torch.bfloat16, dev)
        self.r_buf, rs = _flat_views(self.specs, torch.int16, dev)
        self.g_buf, gs = _flat_views(self.specs, torch.bfloat16, dev)
        self.m_buf, ms = _flat_views(self.specs, torch.float32, dev)
        self.v_buf, vs = _flat_views(self.specs, torch.float32, dev)
        for i, (h, r, g, s) in enumerate(zip(hs, rs, gs, self.specs)):
            if "norm" in s.name:
                h.fill_(1.0)
            else:
                hi, rem = synth.bf16_params_with_remainders(s.numel, 0.02, seed + i, dev)
                h.copy_(hi)
                r.copy_(rem)
                del hi, rem
            g.copy_(synth.normal(s.numel, 1e-4, synth.grad_seed(seed, 0, i), dev, torch.bfloat16))
        self.opt = FusedAdamW(hs, gs, ms, vs, [s.wd for s in self.specs], mode="bf16_rem",
                              param_rems=rs)
        self._views = (hs, rs, gs, ms, vs)
        self.lr = torch.tensor([3e-4], dtype=torch.float32, device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream().cuda_stream
        self.dtype = "f32 (bf16+int16 params)"
        self.config = Llama3.describe()

    @classmethod
    def describe(cls, seed=5):
        import synth
        specs = synth.llama3_8b()
        return {"workload": "Llama-3-8B param list, bf16 params + int16 remainders, bf16 grads, "
                            "fp32 m and v, lr 3e-4 from a device tensor, wd 0.1",
                "tensors": len(specs), "numel": synth.total_numel(specs),
                "bytes_per_param": Llama3.bytes_per_param, "grad_dtype": "bf16",
                "state_dtype": "f32", "param_dtype": "bf16 + int16 remainder",
                "l2": "no flush: 209 GB moved per step, larger than the 126 MB L2"}

    def step(self, i):
        self.C.adamw_step(self.opt.plan, self.lr.data_ptr(), self.step_dev.data_ptr(), 0.9, 0.999,
                          1e-8, None, None, self.stream)

    def e2e_setup(self, group=1 << 27, ring=3):
        """Groups of `group` consecutive elements of the flat buffers (the padding
        between tensors included in the copies), each stepped by a plan over the
        slices of the tensors it covers (PipelinedE2E with a ring)."""
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW
        hs, rs, gs, ms, vs = self._views
        base = self.h_buf.data_ptr()
        spans = [((h.data_ptr() - base) // 2, h.numel()) for h in hs]
        total = self.h_buf.numel()
        groups = []
        for lo in range(0, total, group):
            hi = min(total, lo + group)
            sel = [[], [], [], [], [], []]
            for j, (o, n) in enumerate(spans):
                a, b = max(lo, o), min(hi, o + n)
                if a >= b:
                    continue
                for lst, t in zip(sel, (hs[j], rs[j], gs[j], ms[j], vs[j])):
                    lst.append(t[a - o:b - o])
                sel[5].append(self.specs[j].wd)
            if sel[0]:
                opt = FusedAdamW(sel[0], sel[2], sel[3], sel[4], sel[5], mode="bf16_rem",
                                 param_rems=sel[1])
                groups.append((lo, hi, opt))
        return self._pipeline([self.g_buf], [self.h_buf, self.r_buf], groups, ring=ring)

    def _group_step(self, opt, i, step_dev, stream):
        self.C.adamw_step(opt.plan, self.lr.data_ptr(), step_dev.data_ptr(), 0.9, 0.999, 1e-8,
                          None, None, stream)


class MiniLlama3(Workload):
    """Adam-mini on the Llama-3-8B list (bf16 params + int16 remainders, bf16 grads).

    Two launches per step: the block reduction reads g of every tensor with a
    shared v (2 B per element), the update streams p, remainder, g, m (and v
    for the per-element embedding and output tensors)."""
    name = "adam_mini_llama3_8b_bf16_rem"
    launches_per_step = 2

    def __init__(self, seed=5):
        import torch
        import synth
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi
        dev = torch.device("cuda")
        self.C = _capi
        self.specs = synth.llama3_8b()
        self.n_params = synth.total_numel(self.specs)
        blocks = synth.adam_mini_blocks(self.specs, dim=4096, n_heads=32)
        _, hs = _flat_views(self.specs, torch.bfloat16, dev)
        _, rs = _flat_views(self.specs, torch.int16, dev)
        _, gs = _flat_views(self.specs, torch.bfloat16, dev)
        _, ms = _flat_views(self.specs, torch.float32, dev)
        vs = [torch.zeros(s.numel // b, device=dev) for s, b in zip(self.specs, blocks)]
        for i, (h, r, g, s) in enumerate(zip(hs, rs, gs, self.specs)):
            if "norm" in s.name:
                h.fill_(1.0)
            else:
                hi, rem = synth.bf16_params_with_remainders(s.numel, 0.02, seed + i, dev)
                h.copy_(hi)
                r.copy_(rem)
                del hi, rem
            g.copy_(synth.normal(s.numel, 1e-4, synth.grad_seed(seed, 0, i), dev, torch.bfloat16))
        wds = [0.0 if "norm" in s.name else 0.1 for s in self.specs]
        self.opt = FusedAdamW(hs, gs, ms, vs, wds, mode="bf16_rem", param_rems=rs, v_blocks=blocks)
        self._views = (hs, rs, gs, ms, vs)
        self.config = MiniLlama3.describe()
        self.bytes_per_param = self.config["bytes_per_param"]
        self.lr = torch.tensor([3e-4], dtype=torch.float32, device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream().cuda_stream
        self.dtype = "f32 (bf16+int16 params)"

    @classmethod
    def describe(cls, seed=5):
        import synth
        specs = synth.llama3_8b()
        blocks = synth.adam_mini_blocks(specs, dim=4096, n_heads=32)
        n = synth.total_numel(specs)
        n_elem_v = sum(s.numel for s, b in zip(specs, blocks) if b == 1)
        # reduction: g (2) of the shared-v tensors; update: p 2 + rem 2 + g 2 + m 4 read,
        # p 2 + rem 2 + m 4 written; per-element v (embeddings, output) adds 4 + 4
        total = 2 * (n - n_elem_v) + 18 * n + 8 * n_elem_v
        return {"workload": "Adam-mini on the Llama-3-8B param list (v per element for "
                            "embeddings/output, per head for wq/wk, per tensor elsewhere), "
                            "bf16 params + int16 remainders",
                "tensors": len(specs), "numel": n, "v_blocks": len(set(blocks)),
                "bytes_per_param": total / n, "l2": f"no flush: {total / 1e9:.0f} GB moved per step"}

    def step(self, i):
        self.C.adamw_mini_step(self.opt.plan, self.lr.data_ptr(), self.step_dev.data_ptr(), 0.9, 0.999,
                               1e-8, None, None, self.stream)

    def e2e_setup(self):
        return None


class Bf16Rem(Workload):
    """One flat bf16+remainder tensor: a small stand-in for the Llama-3-8B list (profiling)."""
    name = "bf16rem_flat"
    bytes_per_param = 26.0

    def __init__(self, seed=6, numel=0):
        import torch
        import synth
        from adamw_optimizer_step_tensor_gb300 import FusedAdamW, _capi
        dev = torch.device("cuda")
        self.C = _capi
        n = self.n_params = numel or (1 << 26)
        self.h, self.r = synth.bf16_params_with_remainders(n, 0.02, seed, dev)
        self.g = synth.normal(n, 1e-4, seed + 1, dev, torch.bfloat16)
        self.m = torch.zeros(n, device=dev)
        self.v = torch.zeros(n, device=dev)
        self.opt = FusedAdamW([self.h], [self.g], [self.m], [self.v], [0.1], mode="bf16_rem",
                              param_rems=[self.r])
        self.lr = torch.tensor([3e-4], dtype=torch.float32, device=dev)
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream().cuda_stream
        self.dtype = "f32 (bf16+int16 params)"
        self.config = Bf16Rem.describe(numel=numel)

    @classmethod
    def describe(cls, seed=6, numel=0):
        return {"workload": "one flat bf16+remainder tensor, bf16 grads", "tensors": 1,
                "numel": numel or (1 << 26), "bytes_per_param": Bf16Rem.bytes_per_param,
                "l2": "no flush: inputs larger than L2"}

    def step(self, i):
        self.C.adamw_step(self.opt.plan, self.lr.data_ptr(), self.step_dev.data_ptr(), 0.9, 0.999,
                          1e-8, None, None, self.stream)


def _workload_table(numel):
    """name -> (class, constructor arguments); the constructor builds the workload on the
    device, ``describe`` with the same arguments gives its config without a device."""
    return {"gpt2_small": (Gpt2Small, {}), "single": (Single, dict(numel=numel)),
            "amp": (Single, dict(amp=True, numel=numel)), "q8": (Q8, dict(numel=numel)),
            "amp_fused": (Single, dict(amp=True, numel=numel, fused=True)),
            "llama3_8b": (Llama3, {}), "bf16rem": (Bf16Rem, dict(numel=numel)),
            "ademamix_gpt2": (AdemamixGpt2, {}), "lion_gpt2": (LionGpt2, {}),
            "momentum_gpt2": (CoupledGpt2, dict(rule="momentum")),
            "rmsprop_gpt2": (CoupledGpt2, dict(rule="rmsprop")),
            "adagrad_gpt2": (CoupledGpt2, dict(rule="adagrad")),
            "q4": (Q4, dict(numel=numel)), "adam_mini_llama3": (MiniLlama3, {})}


def make_workload(name, numel=0):
    cls, kw = _workload_table(numel)[name]
    return cls(**kw)


def describe_workload(name, numel=0):
    cls, kw = _workload_table(numel)[name]
    return cls.describe(**kw)


# ----------------------------------------------------------------------------- graph replay
def graph_replay_us(w, flush, k=100):
    """Per-step device time of the L2-flushed small workloads without the per-launch
    event floor: k (flush + step) pairs captured in one CUDA graph and replayed, minus
    k flushes captured and replayed the same way, divided by k."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    saved = w.stream
    w.stream = side.cuda_stream
    both, flushes = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(both, stream=side):
            for i in range(k):
                flush.zero_()
                w.step(i)
        with torch.cuda.graph(flushes, stream=side):
            for _ in range(k):
                flush.zero_()
    finally:
        w.stream = saved
    torch.cuda.synchronize()

    def timed(g):
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(5):
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best
    return (timed(both) - timed(flushes)) * 1e3 / k


# ----------------------------------------------------------------------------- CPU timing
def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _sample_table(kind):
    if kind == "second":
        return {k: v[1] for k, v in CPU_SAMPLES_SECOND.items()}
    return CPU_SAMPLES


def _cpu_worker(kind, workload, n, seconds, steps, warmup, barrier, out):
    """One host core: builds its own sample of n elements (its own seeded
    inputs, disjoint from every other worker's), warms up, waits for every
    worker at the barrier, then runs the oracle step either for `seconds` or
    for `steps` calls, and reports (elements stepped, seconds, description)."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    try:
        run, desc = _sample_table(kind)[workload](n)
        for _ in range(max(1, warmup)):
            run()
        barrier.wait()
        t0 = time.perf_counter()
        calls = 0
        while (calls < steps) if steps else (calls < 1 or time.perf_counter() - t0 < seconds):
            run()
            calls += 1
        out.put((n * calls, time.perf_counter() - t0, calls, desc, None))
    except Exception as e:  # reported to the parent, which raises
        barrier.abort()
        out.put((0, 0.0, 0, "", repr(e)))


def time_cpu_all_cores(workload, n, seconds=0.0, steps=0, warmup=1, kind="first"):
    """The oracle on every host core at once: one spawned process per core
    (spawn, so that no CUDA state is inherited), each on its own n-element
    sample; the workers start together after their warm-up.  Returns
    (elements per second over the slowest worker's time, cores, calls per
    worker, seconds, description)."""
    import multiprocessing as mp
    cores = cpu_threads()
    ctx = mp.get_context("spawn")
    barrier, out = ctx.Barrier(cores), ctx.Queue()
    procs = [ctx.Process(target=_cpu_worker,
                         args=(kind, workload, n, seconds, steps, warmup, barrier, out))
             for _ in range(cores)]
    for p in procs:
        p.start()
    res = [out.get() for _ in procs]
    for p in procs:
        p.join()
    errs = [r[4] for r in res if r[4]]
    if errs:
        raise RuntimeError(f"CPU oracle worker failed: {errs[0]}")
    elems = sum(r[0] for r in res)
    dt = max(r[1] for r in res)
    return elems / dt, cores, min(r[2] for r in res), dt, res[0][3]


# ----------------------------------------------------------------------------- main
def run_reference(args, rank, world):
    """The oracle as it stands, on every host core, on a bounded sample of the
    workload: each step is one oracle step per core on that core's own sample."""
    if rank != 0:
        return 0
    make = CPU_SAMPLES[args.workload]
    run, _ = make(1 << 16)                     # calibrate: seconds per element on one core
    t0 = time.perf_counter()
    run()
    per_elem = (time.perf_counter() - t0) / (1 << 16)
    budget = 90.0                              # whole --steps/--warmup run within ~2 minutes
    n = int(budget / max(1, args.steps + args.warmup) / max(per_elem, 1e-12))
    n = max(4096, min(1 << 23, n // 256 * 256))
    value, cores, calls, dt, desc = time_cpu_all_cores(args.workload, n, steps=max(1, args.steps),
                                                       warmup=args.warmup)
    steps = max(1, args.steps)
    sample = (f"{desc}, on each of {cores} host cores (one process per core, disjoint samples: "
              f"{n * cores} elements per step); numpy")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": args.warmup, "ms_per_step": dt / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": REFERENCE_DTYPE.get(args.workload, "f64"), "data": "synthetic",
            "config": dict(describe_workload(args.workload, args.numel), parallelism="1 GPU"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    w = make_workload(args.workload, args.numel)
    if args.no_l2_flush and w.flush_l2:
        w.flush_l2 = False
        w.config = dict(w.config, l2="not flushed: the inputs stay resident in the 126 MB L2 "
                                     "between timed launches (an L2-resident rate, not HBM)")
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda") if w.flush_l2 else None

    for i in range(max(3, args.warmup)):
        w.step(i)
    torch.cuda.synchronize()

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_begin = time.time()
    region0.record(stream)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        w.step(args.warmup + i)
        ends[i].record(stream)
    region1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    barrier(world)
    time.sleep(0.3)
    clocks.stop()
    clk = clocks.summary(t_begin, t_end)

    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    region_ms = region0.elapsed_time(region1)
    step_ms = sum(launch_ms) / K if flush is not None else region_ms / K
    step_ms = max_over_ranks(step_ms, world)
    value = w.n_params * world / (step_ms * 1e-3)
    kernel_ms = statistics.mean(launch_ms)
    alg_bytes = w.bytes_per_param * w.n_params
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    peak, peak_src = measured_peak()

    graph = None
    if flush is not None:
        try:
            us = graph_replay_us(w, flush)
            graph = {"us_per_step": us, "achieved_gbs": alg_bytes / (us * 1e-6) / 1e9,
                     "frac": alg_bytes / (us * 1e-6) / 1e9 / peak,
                     "what": "100 (L2 flush + step) pairs in one CUDA graph, replayed; 100 flushes "
                             "replayed alone subtracted: the step without the per-launch event floor"}
        except RuntimeError as e:     # a launch that stream capture does not take
            torch.cuda.synchronize()
            graph = {"us_per_step": None, "note": f"not captured: {str(e).splitlines()[0][:160]}"}

    # ---- end to end through the C ABI with pinned host buffers
    e2e = None
    n_e2e = min(args.e2e_steps, getattr(w, "e2e_steps", args.e2e_steps))
    setup = w.e2e_setup() if hasattr(w, "e2e_setup") and n_e2e > 0 else None
    if setup is not None:
        h2d, d2h = setup
        begin = getattr(w, "e2e_begin", None)
        end = getattr(w, "e2e_end", None)
        if begin:
            begin(stream)
        for i in range(getattr(w, "e2e_warmup", 3)):
            w.e2e_step(i)
        if end:
            end(stream)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if begin:
            begin(stream)
        for i in range(n_e2e):
            w.e2e_step(i)
        if end:
            end(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world)
        e2e = {"value": w.n_params * world / (e2e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "ms_per_step": e2e_ms, "copies_declared": True,
               "what": getattr(w, "e2e_what",
                               "pinned-host grads -> device, adamw_step, updated params -> pinned host")}
    else:
        e2e = {"value": None, "unit": UNIT, "h2d_bytes_per_step": None, "d2h_bytes_per_step": None,
               "note": "this workload has no host-offload arm, or --e2e-steps 0"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = 1 << 21
        v, cores, calls, dt, desc = time_cpu_all_cores(args.workload, n, seconds=args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{desc}, on each of {cores} host cores (one process per core, disjoint "
                         f"samples); {calls}+ steps per core in {dt:.1f} s; numpy"}
        if args.workload in CPU_SAMPLES_SECOND:
            label = CPU_SAMPLES_SECOND[args.workload][0]
            v, cores, calls, dt, desc = time_cpu_all_cores(args.workload, n,
                                                           seconds=args.cpu_seconds / 2,
                                                           kind="second")
            cpu[label] = {"value": v, "unit": UNIT, "cores": cores,
                          "sample": f"{desc}, on each of {cores} host cores; {calls}+ steps per "
                                    f"core in {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(w.config, parallelism=f"replicas x{world}" if world > 1 else "1 GPU"),
            "achieved_hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": ncu_traffic(args.workload),
                         "peak_source": peak_src, "kernel_ms": kernel_ms,
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "nominal_peak": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                         "issue": issue_roofline(args.workload, w.n_params / (kernel_ms * 1e-3),
                                                 (clk or {}).get("sm_mhz"))},
            "e2e": e2e,
            "gpu_launches": K * w.launches_per_step,
            **({"graph_replay": graph} if graph else {}),
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
