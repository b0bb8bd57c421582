"""The design notes and the README name files that exist (CPU only).

Every back-quoted repository path in README.md (tests, kernels,
oracle modules, headers, profiles) must point at a file or directory of the
repository, and every bench workload the measurement table quotes must be one
``bench.py --workload`` accepts; stale names in the documentation are caught
here rather than by a reader.
"""

import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PREFIXES = ("tests/", "csrc/", "oracle/", "include/", "profiles/", "synth/",
            "adamw_optimizer_step_tensor_gb300/")


def _paths(text):
    for tok in re.findall(r"`([^`\s]+)`", text):
        tok = tok.rstrip(".,;:")
        if tok.startswith(PREFIXES) and "*" not in tok and "<" not in tok:
            yield tok.split("::")[0]


def _exists(path):
    for base in (ROOT, os.path.join(ROOT, "adamw_optimizer_step_tensor_gb300")):
        if os.path.exists(os.path.join(base, path)):
            return True
    return False


def test_documented_paths_exist():
    missing = []
    for doc in ("DESIGN.md", "README.md"):
        with open(os.path.join(ROOT, doc)) as f:
            text = f.read()
        missing += [(doc, p) for p in _paths(text) if not _exists(p)]
    assert not missing, missing


def test_documented_workloads_exist():
    with open(os.path.join(ROOT, "DESIGN.md")) as f:
        text = f.read()
    names = set(re.findall(r"--workload ([a-z0-9_]+)", text))
    assert names
    assert names <= set(bench._workload_table(0)), names - set(bench._workload_table(0))
