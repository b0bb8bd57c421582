// lane_tables.cuh -- bank-conflict-free code-table lookups for the 8-bit and
// 4-bit steps.
//
// A warp looks up 32 unrelated codes at once.  With a single copy of a table
// in shared memory, lanes whose entries fall in the same bank at different
// addresses are served one after another: 32 random codes of a 256-entry
// table take about 3.5 passes of the shared-memory pipe, and those passes, not
// HBM, bounded the 8-bit step.  Here the map values and the thresholds are
// stored once per lane -- entry k of lane l at word 32k + l -- so lane l only
// ever reads bank l and every lookup is a single pass.  The bucket tables
// (one byte per bucket, 3201 buckets per sign and map) stay single copies:
// 32 copies of them would not fit.
//
// The search itself is the one of nearest_code: the bucket of |x| gives the
// lowest code lo any x of the bucket can have, and code = lo + #{r < R :
// thr[lo + r] <= x}.
#pragma once

#include <cstdint>

#include "internal.h"
#include "step_common.cuh"

namespace adamw {
namespace {

template <int N>   // codes per map: 256 (8-bit) or 16 (4-bit)
struct LaneTables {
  float value[2][N][32];                // [map][code][lane]; map 0 signed (m), 1 unsigned (v)
  float thr[2][N + kMaxRefine][32];     // thresholds, +inf past the last one
  uint8_t lo_pos[2][kBuckets];
  uint8_t lo_neg[kBuckets];             // the signed map's lowest codes of x <= 0
};

// Expand the plan's compact tables into the lane-private layout; every
// thread of the CTA takes part, and the caller synchronises afterwards.
template <int N>
__device__ __forceinline__ void fill_lane_tables(LaneTables<N>& lt, const QTables* qt) {
  const int nt = blockDim.x;
  float* const val = &lt.value[0][0][0];
  for (int i = threadIdx.x; i < 2 * N * 32; i += nt)
    val[i] = qt->map[i / (N * 32)].value[(i / 32) % N];
  float* const thr = &lt.thr[0][0][0];
  for (int i = threadIdx.x; i < 2 * (N + kMaxRefine) * 32; i += nt)
    thr[i] = qt->map[i / ((N + kMaxRefine) * 32)].thr[(i / 32) % (N + kMaxRefine)];
  for (int i = threadIdx.x; i < kBuckets; i += nt) {
    lt.lo_pos[0][i] = qt->map[0].lo_pos[i];
    lt.lo_pos[1][i] = qt->map[1].lo_pos[i];
    lt.lo_neg[i] = qt->map[0].lo_neg[i];
  }
}

// Nearest code of a normalised x in map MAP (0: signed m map, 1: unsigned v
// map, whose inputs are never negative: a NaN of either sign reaches the last
// bucket, whose lowest code is 0 and whose thresholds never compare true).
template <int N, int MAP, int R>
__device__ __forceinline__ uint32_t lane_nearest(const LaneTables<N>& lt, float x, int lane) {
  const uint32_t b = __float_as_uint(x);
  const int k = bucket_of(b & 0x7FFFFFFFu);
  const uint8_t* const tab = (MAP == 0 && (b >> 31)) ? lt.lo_neg : lt.lo_pos[MAP];
  const uint32_t lo = tab[k];
  uint32_t c = lo;
#pragma unroll
  for (int r = 0; r < R; ++r) c += (lt.thr[MAP][lo + r][lane] <= x) ? 1u : 0u;
  return c;
}

// Codes of the 8 values one lane owns, given the block constants (see
// quant8: the branches are warp- or half-warp-uniform; x * 1 is exact).
template <int N, int MAP, int R>
__device__ __forceinline__ void lane_quant8(const LaneTables<N>& lt, const float (&x)[8],
                                            const BlockNorm& n, uint32_t zero_code, int lane,
                                            uint32_t (&q)[8]) {
  if (n.bits == 0u) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = zero_code;
  } else if (n.scale == 1.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = lane_nearest<N, MAP, R>(lt, __fmul_rn(x[i], n.inv), lane);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      q[i] = lane_nearest<N, MAP, R>(lt, __fmul_rn(__fmul_rn(x[i], n.scale), n.inv), lane);
  }
}

}  // namespace
}  // namespace adamw
