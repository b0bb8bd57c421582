// bulk_kernels.cu -- the fp32 and bf16+remainder steps (AdamW, AdEMAMix, Lion,
// momentum / RMSprop / Adagrad with coupled L2, and the element update of
// Adam-mini) with bulk-async staging.
//
// One CTA per SM (two for RMSprop and Adagrad): a producer warp streams each
// 2048-element tile of every input the rule reads (p [+ remainder], g, m, and
// v / the slow EMA where it has them) into a ring of shared-memory stages with
// cp.async.bulk (the TMA engine, completion counted on an mbarrier per stage),
// and sixteen consumer warps update the tile from shared memory and store the
// results straight to global memory.  Many tiles are in flight per SM without
// holding them in registers, which is what an HBM-bound stream needs.
//
// Every wait on an mbarrier is bounded: after kWaitLimitNs (2 s of
// %globaltimer) the waiting thread records a fault code in the plan's scratch
// word and leaves; a producer that gives up first waits, again bounded, for
// the copies it already issued so none lands in freed shared memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "step_common.cuh"
#include "async_copy.cuh"

namespace adamw {
namespace {

constexpr int kConsumers = kBulkConsumers;     // consumer threads (16 warps)
constexpr int kTile = kConsumers * 4;           // elements per stage: 4 per consumer thread
static_assert(kTile % kVec == 0, "bulk copies move whole 8-element groups");
// Byte layout of one stage: p, rem (bf16 mode), g, m, v (not Lion), m2
// (AdEMAMix) -- each kTile elements.
template <adamw_mode MODE, typename GT, int ALGO>
struct Stage {
  static constexpr bool kV = algo_two_state(ALGO);
  static constexpr bool kM2 = ALGO == kAlgoAdemamix;
  static constexpr int kP = MODE == ADAMW_MODE_FP32 ? 4 : 2;
  static constexpr int kG = sizeof(GT);
  static constexpr int oP = 0;
  static constexpr int oR = oP + kTile * kP;
  static constexpr int oG = oR + (MODE == ADAMW_MODE_BF16_REM ? kTile * 2 : 0);
  static constexpr int oM = oG + kTile * kG;
  static constexpr int oV = oM + kTile * 4;
  static constexpr int oM2 = oV + (kV ? kTile * 4 : 0);
  static constexpr int kBytes = oM2 + (kM2 ? kTile * 4 : 0);
  // bytes moved per element in bulk
  static constexpr int kPerElem =
      kP + (MODE == ADAMW_MODE_BF16_REM ? 2 : 0) + kG + 4 + (kV ? 4 : 0) + (kM2 ? 4 : 0);
  static_assert(kBytes % 128 == 0, "stages stay 128-byte aligned");
};

// Resident CTAs per SM the register budget targets, and pipeline stages per
// CTA.  Measured on GB300 (GPT-2 list, fp32): AdamW with 16 consumer warps and
// 3 stages moved 98% of the copy bandwidth (8 warps x 6 stages 91%, 16 x 4-5
// stages 97%, 16 x 2 stages 96%, 24-30 warps 96-97%); Lion 3 stages 0.368 ms,
// 4 stages 0.371, 2 stages 0.419.  RMSprop and Adagrad do a square root and a
// division for every 20 bytes and hide their latency with two CTAs per SM of
// two stages each (0.448 ms at 1 x 3, 0.398 at 2 x 3, 0.377 at 2 x 2, 0.412 at
// 2 x 4); Lion and momentum, without them, run faster at one CTA (0.371 vs
// 0.384 ms).
template <int ALGO> struct AlgoTune {
  static constexpr bool sqrt_div = ALGO == kAlgoRmsprop || ALGO == kAlgoAdagrad;
  static constexpr int ctas = sqrt_div ? 2 : 1;
  static constexpr int stages = sqrt_div ? 2 : 3;
};

template <adamw_mode MODE, typename GT, int ALGO>
constexpr int bulk_smem_bytes() {
  return AlgoTune<ALGO>::stages * Stage<MODE, GT, ALGO>::kBytes + 2 * AlgoTune<ALGO>::stages * 8;
}

__device__ __forceinline__ void fault(const StepArgs& a, uint32_t code) {
  atomicOr(&a.scratch->fault, code);
}

// The producer: one thread issues the bulk copies of every tile of this CTA.
template <adamw_mode MODE, typename GT, int ALGO>
__device__ void produce(const StepArgs& a, unsigned char* ring, uint64_t* full, uint64_t* empty) {
  using L = Stage<MODE, GT, ALGO>;
  constexpr int S = AlgoTune<ALGO>::stages;
  uint32_t i = 0;
  bool ok = true;
  for (int64_t c = blockIdx.x; ok && c < a.n_chunks; c += gridDim.x) {
    const Chunk ch = a.chunks[c];
    const TensorDesc td = a.tensors[ch.tensor];
    // Adam-mini chunks of a shared-v block stream no v
    const bool copy_v = L::kV && !(ALGO == kAlgoMini && a.chunk_blk[c] >= 0);
    const uint32_t per_elem = L::kPerElem - ((L::kV && !copy_v) ? 4u : 0u);
    for (int k = 0; k * kTile < ch.len; ++k, ++i) {
      const uint32_t s = i % S;
      if (!mbar_wait(&empty[s], ((i / S) & 1u) ^ 1u)) {
        fault(a, 1u);
        ok = false;
        break;
      }
      const int len = min(kTile, ch.len - k * kTile);
      const int nb = td.vec_ok ? (len & ~(kVec - 1)) : 0;  // elements moved in bulk
      const int64_t e = ch.start + static_cast<int64_t>(k) * kTile;
      unsigned char* st = ring + static_cast<size_t>(s) * L::kBytes;
      const uint32_t bytes = nb * per_elem;
      mbar_expect_tx(&full[s], bytes);
      if (nb > 0) {
        bulk_g2s(st + L::oP, static_cast<const unsigned char*>(td.p) + e * L::kP, nb * L::kP, &full[s]);
        if (MODE == ADAMW_MODE_BF16_REM)
          bulk_g2s(st + L::oR, td.rem + e, nb * 2, &full[s]);
        bulk_g2s(st + L::oG, static_cast<const unsigned char*>(td.g) + e * L::kG, nb * L::kG, &full[s]);
        bulk_g2s(st + L::oM, static_cast<const float*>(td.m) + e, nb * 4, &full[s]);
        if (copy_v) bulk_g2s(st + L::oV, static_cast<const float*>(td.v) + e, nb * 4, &full[s]);
        if (L::kM2) bulk_g2s(st + L::oM2, static_cast<const float*>(td.m2) + e, nb * 4, &full[s]);
      }
    }
  }
  if (!ok) {
    // drain: every stage issued in the last S tiles completes on its own
    for (uint32_t j = (i > S ? i - S : 0); j < i; ++j)
      if (!mbar_wait(&full[j % S], (j / S) & 1u)) fault(a, 4u);
  }
}

// Four consecutive elements [j, j+4) of a tile from shared memory.
template <adamw_mode MODE, typename GT, int ALGO>
__device__ __forceinline__ void load4_smem(const unsigned char* st, int j, float (&p)[4],
                                           float (&g)[4], float (&m)[4], float (&v)[4]) {
  using L = Stage<MODE, GT, ALGO>;
  if (MODE == ADAMW_MODE_FP32) {
    const float4 x = *reinterpret_cast<const float4*>(st + L::oP + j * 4);
    p[0] = x.x; p[1] = x.y; p[2] = x.z; p[3] = x.w;
  } else {
    const uint2 h = *reinterpret_cast<const uint2*>(st + L::oP + j * 2);
    const uint2 r = *reinterpret_cast<const uint2*>(st + L::oR + j * 2);
    p[0] = rem_join(h.x & 0xFFFFu, r.x & 0xFFFFu);
    p[1] = rem_join(h.x >> 16, r.x >> 16);
    p[2] = rem_join(h.y & 0xFFFFu, r.y & 0xFFFFu);
    p[3] = rem_join(h.y >> 16, r.y >> 16);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) g[q] = grad_from_smem<GT>(st + L::oG, j + q);
  const float4 mm = *reinterpret_cast<const float4*>(st + L::oM + j * 4);
  m[0] = mm.x; m[1] = mm.y; m[2] = mm.z; m[3] = mm.w;
  if (L::kV) {
    const float4 vv = *reinterpret_cast<const float4*>(st + L::oV + j * 4);
    v[0] = vv.x; v[1] = vv.y; v[2] = vv.z; v[3] = vv.w;
  }
}

template <adamw_mode MODE, bool kV>
__device__ __forceinline__ void store4(const TensorDesc& td, int64_t e, const float (&p)[4],
                                       const float (&m)[4], const float (&v)[4]) {
  if (MODE == ADAMW_MODE_FP32) {
    __stcs(reinterpret_cast<float4*>(static_cast<float*>(td.p) + e), make_float4(p[0], p[1], p[2], p[3]));
  } else {
    uint32_t h0, r0, h1, r1, h2, r2, h3, r3;
    rem_split(p[0], h0, r0);
    rem_split(p[1], h1, r1);
    rem_split(p[2], h2, r2);
    rem_split(p[3], h3, r3);
    __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(td.p) + e),
           make_uint2(h0 | (h1 << 16), h2 | (h3 << 16)));
    __stcs(reinterpret_cast<uint2*>(td.rem + e), make_uint2(r0 | (r1 << 16), r2 | (r3 << 16)));
  }
  __stcs(reinterpret_cast<float4*>(static_cast<float*>(td.m) + e), make_float4(m[0], m[1], m[2], m[3]));
  if (kV)
    __stcs(reinterpret_cast<float4*>(static_cast<float*>(td.v) + e), make_float4(v[0], v[1], v[2], v[3]));
}

template <adamw_mode MODE, typename GT, int ALGO>
__global__ void __launch_bounds__(kBulkThreads, AlgoTune<ALGO>::ctas) step_bulk_kernel(const StepArgs a) {
  using L = Stage<MODE, GT, ALGO>;
  constexpr int S = AlgoTune<ALGO>::stages;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* ring = smem_raw;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + S * L::kBytes);
  uint64_t* empty = full + S;
  __shared__ Scal s_sc;
  __shared__ int s_skip;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);                     // the producer's arrive.expect_tx
      mbar_init(&empty[s], kConsumers / 32);      // one arrive per consumer warp
    }
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();

  if (threadIdx.x >= kConsumers) {
    // producer warp: one lane issues; the skip flag is read here too, so that
    // no copy is issued for a skipped step
    if (threadIdx.x == kConsumers) {
      const bool skip = a.found_inf != nullptr && *a.found_inf != 0.0f;
      if (!skip) produce<MODE, GT, ALGO>(a, ring, full, empty);
    }
    return;
  }

  int t = 0;
  if (threadIdx.x == 0) s_skip = prologue(a, s_sc, t);
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");   // consumers only
  if (s_skip) return;
  const Scal s = s_sc;
  if (threadIdx.x == 0) take_ticket(a, t);
  const int lane = threadIdx.x & 31;

  uint32_t i = 0;
  for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
    const Chunk ch = a.chunks[c];
    const TensorDesc td = a.tensors[ch.tensor];
    // the parameter's decay factor; the coupled rules take wd itself, Adam-mini
    // decays only when wd > 0
    const float decay = algo_coupled(ALGO) ? td.wd
                        : (ALGO == kAlgoMini && !(td.wd > 0.0f)) ? 1.0f
                        : __fsub_rn(1.0f, __fmul_rn(s.lr, td.wd));
    int32_t mini_blk = -1;
    float mini_r = 0.0f;
    if (ALGO == kAlgoMini) {
      mini_blk = a.chunk_blk[c];
      if (mini_blk >= 0) mini_r = a.blk_r[mini_blk];
    }
    for (int k = 0; k * kTile < ch.len; ++k, ++i) {
      const uint32_t st_i = i % S;
      if (!mbar_wait(&full[st_i], (i / S) & 1u)) {
        fault(a, 2u);
        return;
      }
      const int len = min(kTile, ch.len - k * kTile);
      const int nb = td.vec_ok ? (len & ~(kVec - 1)) : 0;
      const int64_t e0 = ch.start + static_cast<int64_t>(k) * kTile;
      const unsigned char* st = ring + static_cast<size_t>(st_i) * L::kBytes;
      // thread t owns elements [4t, 4t+4) of the tile: conflict-free 16-byte smem reads
      {
        const int j = threadIdx.x * 4;
        if (j + 4 <= nb) {
          float p[4], g[4], m[4], v[4];
          load4_smem<MODE, GT, ALGO>(st, j, p, g, m, v);
          if (ALGO == kAlgoMini && mini_blk >= 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) update_mini(p[q], g[q], m[q], mini_r, s, decay);
          } else if (algo_coupled(ALGO)) {
#pragma unroll
            for (int q = 0; q < 4; ++q) update_coupled<ALGO>(p[q], g[q], m[q], s, decay);
          } else if (ALGO == kAlgoAdemamix) {
            const float4 w = *reinterpret_cast<const float4*>(st + L::oM2 + j * 4);
            float m2[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) update_ademamix(p[q], g[q], m[q], m2[q], v[q], s, decay);
            __stcs(reinterpret_cast<float4*>(static_cast<float*>(td.m2) + e0 + j),
                   make_float4(m2[0], m2[1], m2[2], m2[3]));
          } else if (ALGO == kAlgoLion) {
#pragma unroll
            for (int q = 0; q < 4; ++q) update_lion(p[q], g[q], m[q], s, decay);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) update(p[q], g[q], m[q], v[q], s, decay);
          }
          if (ALGO == kAlgoMini && mini_blk >= 0)
            store4<MODE, false>(td, e0 + j, p, m, v);
          else
            store4<MODE, L::kV>(td, e0 + j, p, m, v);
        } else if (j < len) {
          update_scalar<MODE, GT, ALGO>(td, e0 + j, min(4, len - j), s, decay, mini_r, mini_blk >= 0);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st_i]);
    }
  }
}

template <adamw_mode MODE, typename GT, int ALGO>
cudaError_t launch_one(const StepArgs& a, int grid, cudaStream_t st) {
  step_bulk_kernel<MODE, GT, ALGO><<<grid, kBulkThreads, bulk_smem_bytes<MODE, GT, ALGO>(), st>>>(a);
  return cudaGetLastError();
}

template <adamw_mode MODE, typename GT, int ALGO>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(step_bulk_kernel<MODE, GT, ALGO>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              bulk_smem_bytes<MODE, GT, ALGO>());
}

template <adamw_mode MODE, typename GT, int ALGO>
cudaError_t occupancy_one(int* blocks) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, step_bulk_kernel<MODE, GT, ALGO>,
                                                       kBulkThreads, bulk_smem_bytes<MODE, GT, ALGO>());
}

template <adamw_mode MODE, typename GT>
cudaError_t launch_algo(const StepArgs& a, int grid, cudaStream_t st, int algo) {
  switch (algo) {
    case kAlgoAdamW: return launch_one<MODE, GT, kAlgoAdamW>(a, grid, st);
    case kAlgoAdemamix: return launch_one<MODE, GT, kAlgoAdemamix>(a, grid, st);
    case kAlgoLion: return launch_one<MODE, GT, kAlgoLion>(a, grid, st);
    case kAlgoMomentum: return launch_one<MODE, GT, kAlgoMomentum>(a, grid, st);
    case kAlgoRmsprop: return launch_one<MODE, GT, kAlgoRmsprop>(a, grid, st);
    case kAlgoAdagrad: return launch_one<MODE, GT, kAlgoAdagrad>(a, grid, st);
    case kAlgoMini: return launch_one<MODE, GT, kAlgoMini>(a, grid, st);
  }
  return cudaErrorInvalidValue;
}

template <adamw_mode MODE, typename GT>
cudaError_t prepare_algo(int algo) {
  switch (algo) {
    case kAlgoAdamW: return prepare_one<MODE, GT, kAlgoAdamW>();
    case kAlgoAdemamix: return prepare_one<MODE, GT, kAlgoAdemamix>();
    case kAlgoLion: return prepare_one<MODE, GT, kAlgoLion>();
    case kAlgoMomentum: return prepare_one<MODE, GT, kAlgoMomentum>();
    case kAlgoRmsprop: return prepare_one<MODE, GT, kAlgoRmsprop>();
    case kAlgoAdagrad: return prepare_one<MODE, GT, kAlgoAdagrad>();
    case kAlgoMini: return prepare_one<MODE, GT, kAlgoMini>();
  }
  return cudaErrorInvalidValue;
}

template <typename GT>
cudaError_t launch_bulk_mode(adamw_mode mode, const StepArgs& a, int grid, cudaStream_t st,
                             int algo) {
  if (mode == ADAMW_MODE_FP32) return launch_algo<ADAMW_MODE_FP32, GT>(a, grid, st, algo);
  return launch_algo<ADAMW_MODE_BF16_REM, GT>(a, grid, st, algo);
}

template <typename GT>
cudaError_t prepare_bulk_mode(adamw_mode mode, int algo) {
  if (mode == ADAMW_MODE_FP32) return prepare_algo<ADAMW_MODE_FP32, GT>(algo);
  return prepare_algo<ADAMW_MODE_BF16_REM, GT>(algo);
}

// Self-test of the bounded wait: one thread waits on an mbarrier phase that
// nothing completes; the wait must give up after limit_ns and report it.
__device__ uint32_t g_selftest_fault;
__device__ unsigned long long g_selftest_ns;

__global__ void wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  const uint64_t t0 = global_ns();
  const bool done = mbar_wait(&bar, 0u, limit_ns);   // phase 0 never completes
  g_selftest_ns = global_ns() - t0;
  g_selftest_fault = done ? 0u : 1u;
}

}  // namespace

cudaError_t run_wait_selftest(int limit_us, cudaStream_t s, uint32_t* fault_bits,
                              double* waited_ms) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(limit_us) * 1000ull);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  unsigned long long ns = 0;
  if ((e = cudaMemcpyFromSymbol(fault_bits, g_selftest_fault, sizeof(uint32_t))) != cudaSuccess)
    return e;
  if ((e = cudaMemcpyFromSymbol(&ns, g_selftest_ns, sizeof(ns))) != cudaSuccess) return e;
  *waited_ms = static_cast<double>(ns) * 1e-6;
  return cudaSuccess;
}

cudaError_t launch_step_bulk(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                             cudaStream_t s, int algo) {
  switch (gdt) {
    case ADAMW_F32: return launch_bulk_mode<float>(mode, a, grid, s, algo);
    case ADAMW_F16: return launch_bulk_mode<__half>(mode, a, grid, s, algo);
    case ADAMW_BF16: return launch_bulk_mode<__nv_bfloat16>(mode, a, grid, s, algo);
  }
  return cudaErrorInvalidValue;
}

cudaError_t bulk_occupancy_sqrt_div(adamw_mode mode, adamw_dtype gdt, int* blocks) {
  const bool f = mode == ADAMW_MODE_FP32;
  switch (gdt) {
    case ADAMW_F32:
      return f ? occupancy_one<ADAMW_MODE_FP32, float, kAlgoRmsprop>(blocks)
               : occupancy_one<ADAMW_MODE_BF16_REM, float, kAlgoRmsprop>(blocks);
    case ADAMW_F16:
      return f ? occupancy_one<ADAMW_MODE_FP32, __half, kAlgoRmsprop>(blocks)
               : occupancy_one<ADAMW_MODE_BF16_REM, __half, kAlgoRmsprop>(blocks);
    case ADAMW_BF16:
      return f ? occupancy_one<ADAMW_MODE_FP32, __nv_bfloat16, kAlgoRmsprop>(blocks)
               : occupancy_one<ADAMW_MODE_BF16_REM, __nv_bfloat16, kAlgoRmsprop>(blocks);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_step_bulk(adamw_mode mode, adamw_dtype gdt, int algo) {
  switch (gdt) {
    case ADAMW_F32: return prepare_bulk_mode<float>(mode, algo);
    case ADAMW_F16: return prepare_bulk_mode<__half>(mode, algo);
    case ADAMW_BF16: return prepare_bulk_mode<__nv_bfloat16>(mode, algo);
  }
  return cudaErrorInvalidValue;
}

}  // namespace adamw
