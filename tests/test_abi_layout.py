"""The Python binding and the C header agree on the ABI (CPU only).

A C program compiled against ``include/adamw.h`` prints the size and field
offsets of ``adamw_tensor`` and the values of every enum and define the
binding mirrors; the ctypes structure and constants of ``_capi`` must match
them exactly -- a mismatch would hand the library shifted pointers without
any error.
"""

import ctypes
import os
import shutil
import subprocess

import pytest

from adamw_optimizer_step_tensor_gb300 import _capi as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FIELDS = ["param", "param_rem", "grad", "exp_avg", "exp_avg_sq", "absmax_m", "absmax_v",
          "numel", "weight_decay", "exp_avg_slow"]
CONSTANTS = {
    "ADAMW_OK": C.OK, "ADAMW_EINVAL": C.EINVAL, "ADAMW_EALIGN": C.EALIGN,
    "ADAMW_EDTYPE": C.EDTYPE, "ADAMW_ENOMEM": C.ENOMEM, "ADAMW_ECUDA": C.ECUDA,
    "ADAMW_EUNSUPPORTED": C.EUNSUPPORTED, "ADAMW_ETIMEOUT": C.ETIMEOUT,
    "ADAMW_F32": C.F32, "ADAMW_F16": C.F16, "ADAMW_BF16": C.BF16,
    "ADAMW_MODE_FP32": C.MODE_FP32, "ADAMW_MODE_BF16_REM": C.MODE_BF16_REM,
    "ADAMW_MODE_Q8": C.MODE_Q8, "ADAMW_MODE_Q4": C.MODE_Q4,
    "ADAMW_Q8_BLOCK": C.Q8_BLOCK, "ADAMW_Q4_BLOCK": C.Q4_BLOCK,
    "ADAMW_RULE_MOMENTUM": C.RULES["momentum"], "ADAMW_RULE_RMSPROP": C.RULES["rmsprop"],
    "ADAMW_RULE_ADAGRAD": C.RULES["adagrad"],
}


@pytest.fixture(scope="module")
def c_view(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    d = tmp_path_factory.mktemp("abi")
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "adamw.h"', "int main(void) {",
             '  printf("size %zu\\n", sizeof(adamw_tensor));']
    lines += [f'  printf("off {f} %zu\\n", offsetof(adamw_tensor, {f}));' for f in FIELDS]
    lines += [f'  printf("const {k} %lld\\n", (long long){k});' for k in CONSTANTS]
    lines += ['  printf("const ADAMW_ABI_VERSION %lld\\n", (long long)ADAMW_ABI_VERSION);',
              "  return 0;", "}"]
    src = d / "abi.c"
    src.write_text("\n".join(lines) + "\n")
    exe = d / "abi"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    view = {"off": {}, "const": {}}
    for line in out.splitlines():
        kind, *rest = line.split()
        if kind == "size":
            view["size"] = int(rest[0])
        else:
            view[kind][rest[0]] = int(rest[1])
    return view


def test_tensor_record_layout(c_view):
    assert [f for f, _ in C.adamw_tensor._fields_] == FIELDS
    assert ctypes.sizeof(C.adamw_tensor) == c_view["size"]
    for f in FIELDS:
        assert getattr(C.adamw_tensor, f).offset == c_view["off"][f], f


def test_constants(c_view):
    for k, v in CONSTANTS.items():
        assert c_view["const"][k] == v, k
    assert c_view["const"]["ADAMW_ABI_VERSION"] == 3
