"""The committed ncu summaries belong to the kernels they describe.

Every ``profiles/step_kernel_<workload>.md`` records the hash of the source
files of its kernel; bench.py reports the summary's DRAM traffic and warp
instructions per element only while that hash matches the current sources.
A kernel edited without a new capture would silently drop both figures from
the bench line; this test catches that on the CPU.  Each summary also states
the full command that made it, with the clocks left alone.
"""

import glob
import os
import re

import bench


def _summaries():
    paths = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "step_kernel_*.md")))
    assert paths, "no ncu summaries committed"
    return [(os.path.basename(p)[len("step_kernel_"):-len(".md")], open(p).read()) for p in paths]


def test_every_kernel_summary_matches_its_source():
    for workload, txt in _summaries():
        sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
        assert sha, workload
        assert sha.group(1) == bench.kernel_source_sha(workload), (
            f"{workload}: the kernel's sources changed since its ncu capture")
        assert bench.ncu_traffic(workload) is not None, workload
        assert bench.ncu_figure(workload, "warp_instructions_per_element") is not None, workload


def test_every_summary_names_its_command():
    for workload, txt in _summaries():
        ncu = [line for line in txt.splitlines() if line.startswith("    ncu ")]   # the command block
        assert ncu, workload
        for line in ncu:
            assert "--clock-control none" in line, workload
            assert "python bench.py" in line, workload
