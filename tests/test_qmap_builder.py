"""The library's host-side code-map builder, compiled on the CPU (no GPU).

``csrc/qmap.cpp`` builds the maps and the search tables the 8-bit and 4-bit
kernels use (values, thresholds, per-bucket lowest codes, and the number of
thresholds to compare per lookup).  A small C++ driver compiled with the host
compiler against that file prints them; they must equal, bit for bit, the
oracle's maps and thresholds and the bucket tables rebuilt from their
definition in ``test_bucket_search``.
"""

import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import qmap

from test_bucket_search import N_BUCKETS, tables

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "adamw_optimizer_step_tensor_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include <cstring>
#include "internal.h"
namespace adamw {
void default_maps(float smap[256], float umap[256]);
void default_maps4(float smap[16], float umap[16]);
int build_qmap(const float* value, int n, QMapDev* out);
}
using namespace adamw;
static void dump(const char* name, const float* v, int n) {
  QMapDev t;
  const int r = build_qmap(v, n, &t);
  std::printf("map %s %d %d\n", name, n, r);
  for (int k = 0; k < n; ++k) { unsigned b; std::memcpy(&b, &t.value[k], 4); std::printf("v %u\n", b); }
  for (int k = 0; k < 256 + kMaxRefine; ++k) { unsigned b; std::memcpy(&b, &t.thr[k], 4); std::printf("t %u\n", b); }
  for (int k = 0; k < kBuckets; ++k) std::printf("b %d %d\n", t.lo_pos[k], t.lo_neg[k]);
}
int main() {
  float s8[256], u8[256], s4[16], u4[16];
  default_maps(s8, u8);
  default_maps4(s4, u4);
  dump("s8", s8, 256); dump("u8", u8, 256); dump("s4", s4, 16); dump("u4", u4, 16);
  return 0;
}
"""


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime.h")):
            return os.path.join(d, "include")
    return None


@pytest.fixture(scope="module")
def built(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    d = tmp_path_factory.mktemp("qmap")
    (d / "driver.cpp").write_text(DRIVER)
    exe = d / "driver"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    "-I", inc, str(d / "driver.cpp"), os.path.join(CSRC, "qmap.cpp"), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    maps, cur = {}, None
    for line in out.splitlines():
        f = line.split()
        if f[0] == "map":
            cur = maps[f[1]] = {"n": int(f[2]), "refine": int(f[3]), "v": [], "t": [], "b": []}
        elif f[0] == "b":
            cur["b"].append((int(f[1]), int(f[2])))
        else:
            cur[f[0]].append(int(f[1]))
    return maps


ORACLE = {"s8": qmap.signed_map, "u8": qmap.unsigned_map, "s4": qmap.signed_map4,
          "u4": qmap.unsigned_map4}


@pytest.mark.parametrize("name", sorted(ORACLE))
def test_builder_matches_oracle(built, name):
    m = built[name]
    table = ORACLE[name]()
    n = table.size
    assert m["n"] == n
    assert np.array_equal(np.array(m["v"], np.uint32), table.view(np.uint32))
    thr = qmap.thresholds(table)
    got_thr = np.array(m["t"], np.uint32).view(np.float32)
    assert np.array_equal(got_thr[: n - 1].view(np.uint32), thr.view(np.uint32))
    assert np.all(np.isinf(got_thr[n - 1:]) & (got_thr[n - 1:] > 0))      # +inf padding
    lo_pos, lo_neg, r = tables(thr)
    b = np.array(m["b"])
    assert b.shape == (N_BUCKETS, 2)
    assert np.array_equal(b[:, 0], lo_pos) and np.array_equal(b[:, 1], lo_neg)
    assert max(m["refine"], 1) == r
