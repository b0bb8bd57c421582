// small_kernels.cu -- the fp32 and bf16+remainder AdamW step for plans small
// enough that every CTA's whole share sits in shared memory at once (about
// two million elements or fewer), and its fused non-finite check + step.
//
// At these sizes a step lasts a few microseconds and the launch, the latency
// of the first bytes and the last CTA's tail decide its time, not the
// streaming rate.  So nothing here waits on anything it need not:
//   - the tensor table is a kernel parameter (__grid_constant__): a CTA knows
//     its piece from constant memory, with no dependent global load before its
//     first copy;
//   - every CTA takes exactly one piece of one tensor, and each of its 32 warps
//     a contiguous slice of it; lane 0 of every warp issues the bulk copies of
//     its slice the moment the kernel starts (grads on one mbarrier, then
//     p [+ remainder], m, v on another), right after the warp's own loads of
//     the run-time scalars, which every warp finishes itself: no CTA-wide
//     barrier stands between a warp's data and its arithmetic;
//   - each warp updates its slice as soon as the slice has landed, writes the
//     results back in place in shared memory, and lane 0 streams them out with
//     bulk shared->global copies;
//   - the fused variant scans the raw grads from shared memory as soon as
//     they land (read from HBM once), publishes the CTA's vote, computes the
//     update in place while the other CTAs vote, and only its stores wait for
//     the grid-wide result: one cooperative launch for the check and the step
//     ("FusedAdam & PyTorch Lightning AMP": the fused optimizer unscales and
//     skips on found_inf itself).
//
// The element update is the strict-fp32 sequence of every other step kernel
// (step_common.cuh); ragged tails (< 8 elements of a tensor) and tensors whose
// pointers are not 16-byte aligned go through the scalar path from global
// memory.  Every mbarrier wait is bounded (2 s); a wait that gives up sets a
// fault bit in the plan's scratch word and the CTA stores nothing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "step_common.cuh"
#include "async_copy.cuh"

namespace adamw {
namespace {

constexpr int kSmallWarps = kSmallThreads / 32;

// Bytes per element of the staged streams; the fused variant also keeps the
// results apart from the staged originals (p [+ remainder], m, v).
template <adamw_mode MODE, typename GT, bool FUSED>
struct SmallLayout {
  static constexpr int kP = MODE == ADAMW_MODE_FP32 ? 4 : 2;
  static constexpr int kR = MODE == ADAMW_MODE_BF16_REM ? 2 : 0;
  static constexpr int kG = sizeof(GT);
  static constexpr int kLoad = kP + kR + kG + 8;               // bytes loaded per element
  static constexpr int kPerElem = kLoad + (FUSED ? kP + kR + 8 : 0);
};

__device__ __forceinline__ TensorDesc as_desc(const SmallTensor& t) {
  TensorDesc d{};
  d.p = t.p;
  d.rem = t.rem;
  d.g = t.g;
  d.m = t.m;
  d.v = t.v;
  d.numel = t.numel;
  d.wd = t.wd;
  d.vec_ok = t.vec_ok;
  return d;
}

__device__ __forceinline__ StepArgs as_step_args(const SmallArgs& a, bool with_found_inf) {
  StepArgs s{};
  s.lr = a.lr;
  s.step = a.step;
  s.grad_scale = a.grad_scale;
  s.found_inf = with_found_inf ? a.found_inf : nullptr;
  s.beta1 = a.beta1;
  s.beta2 = a.beta2;
  s.eps = a.eps;
  s.scratch = a.scratch;
  return s;
}

template <adamw_mode MODE, typename GT, bool FUSED>
__global__ void __launch_bounds__(kSmallThreads, 1)
step_small_kernel(const __grid_constant__ SmallArgs a, float* found_inf_out) {
  using L = SmallLayout<MODE, GT, FUSED>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bar_g[kSmallWarps];    // the warp's grads have landed
  __shared__ uint64_t bar_s[kSmallWarps];    // its params and states have landed
  __shared__ int s_bad[kSmallWarps];         // fused: the warp saw a non-finite grad
  __shared__ int s_vote;                     // fused: -1 until the lead warp has the vote
  __shared__ BiasCorr s_next;                // the next step's bias corrections
  // the lead warp, whose slice lands last, takes the CTA's step ticket (and,
  // fused, runs the grid vote) while the other warps compute; the warp before
  // it, whose slice lands next to last, computes the next step's float64 bias
  // corrections while it waits for its data
  constexpr int kLead = kSmallWarps - 1;
  constexpr int kNext = kSmallWarps - 2;
  if (FUSED && threadIdx.x == 0) s_vote = -1;
  if (FUSED) __syncthreads();   // before any memory traffic: costs a few cycles

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's piece: tensor ti, elements [start, start + len)
  int ti = 0;
  while (ti + 1 < a.n_tensors && static_cast<int>(blockIdx.x) >= a.t[ti + 1].first_item) ++ti;
  const SmallTensor& T = a.t[ti];
  const int64_t start = static_cast<int64_t>(blockIdx.x - T.first_item) * T.piece;
  const int len = static_cast<int>(min(static_cast<int64_t>(T.piece), T.numel - start));
  const int nvec = T.vec_ok ? (len & ~(kVec - 1)) : 0;   // elements staged in bulk
  // warp slices of S elements (a multiple of 8: every stream's slice is a
  // whole number of 16-byte words); the slices of one CTA are contiguous
  const int S = (nvec + kSmallWarps * kVec - 1) / (kSmallWarps * kVec) * kVec;
  const int w0 = min(warp * S, nvec);
  const int wn = min(w0 + S, nvec) - w0;
  unsigned char* const base = smem + static_cast<size_t>(warp) * S * L::kPerElem;
  unsigned char* const sP = base;
  unsigned char* const sR = sP + S * L::kP;
  unsigned char* const sG = sR + S * L::kR;
  unsigned char* const sM = sG + S * L::kG;
  unsigned char* const sV = sM + S * 4;
  // where the results go: in place, or (fused) beside the originals, which a
  // skipped step writes back
  unsigned char* const oP = FUSED ? sV + S * 4 : sP;
  unsigned char* const oR = FUSED ? oP + S * L::kP : sR;
  unsigned char* const oM = FUSED ? oR + S * L::kR : sM;
  unsigned char* const oV = FUSED ? oM + S * 4 : sV;
  const int64_t e0 = start + w0;

  // the run-time scalars: every warp loads them itself (the same few words
  // for the whole grid) before its copies go out, so no CTA-wide barrier
  // stands between a warp's data and its arithmetic
  const StepArgs sa = as_step_args(a, !FUSED);
  const RawScalars raw = load_scalars(sa);
  if (lane == 0) {
    mbar_init(&bar_g[warp], 1);
    mbar_init(&bar_s[warp], 1);
    fence_mbar_init();
    if (wn > 0) {
      // grads first: the fused variant scans them while the rest streams in
      mbar_expect_tx(&bar_g[warp], static_cast<uint32_t>(wn) * L::kG);
      bulk_g2s(sG, static_cast<const unsigned char*>(T.g) + e0 * L::kG, wn * L::kG, &bar_g[warp]);
    }
  }
  // fused: every warp's grads are requested before any param or state, so
  // that every CTA can vote early (a barrier before any wait: a few cycles)
  if (FUSED) __syncthreads();
  if (lane == 0) {
    if (wn > 0) {
      mbar_expect_tx(&bar_s[warp], static_cast<uint32_t>(wn) * (L::kLoad - L::kG));
      bulk_g2s(sP, static_cast<const unsigned char*>(T.p) + e0 * L::kP, wn * L::kP, &bar_s[warp]);
      if (MODE == ADAMW_MODE_BF16_REM) bulk_g2s(sR, T.rem + e0, wn * 2, &bar_s[warp]);
      bulk_g2s(sM, T.m + e0, wn * 4, &bar_s[warp]);
      bulk_g2s(sV, T.v + e0, wn * 4, &bar_s[warp]);
    }
  }
  __syncwarp();   // the warp's barriers are initialised before any lane waits on them
  Scal s;
  int t = 0;
  const bool flagged = finish_scalars(sa, raw, s, t);   // found_inf set (plain launch only)
  const float decay = __fsub_rn(1.0f, __fmul_rn(s.lr, T.wd));
  if (warp == kNext && lane == 0 && !flagged) s_next = bias_corrections(a.beta1, a.beta2, next_step(t));
  // fused: the lead takes the launch index now, while the data streams in
  unsigned long long launch = 0;
  if (FUSED && warp == kLead && lane == 0) launch = amp_enter(a.scratch);

  // a slice that does not land in 2 s records fault bit 16 and is not stored;
  // its warp still waits (bounded) so no copy lands in released shared memory
  bool landed = true;
  auto wait_bar = [&](uint64_t* bar) {
    if (wn > 0 && !mbar_wait_suspend(bar, 0u)) {
      if (lane == 0) atomicOr(&a.scratch->fault, 16u);
      mbar_wait_suspend(bar, 0u);
      landed = false;
    }
  };
  if (!FUSED && flagged) {
    wait_bar(&bar_g[warp]);
    wait_bar(&bar_s[warp]);
    return;   // skipped step: nothing is stored, the step counter stays
  }

  // Every warp has read the run-time scalars (*step among them) before it
  // arrives at named barrier 1; the lead warp waits there for all of them.
  // Plain launch: the lead then takes the CTA's ticket at once, so the last
  // CTA's epilogue (the step counter and the next step's float64 bias
  // corrections) runs while the data streams in, not after it.  Fused: each
  // warp first scans the raw grads of its slice as they land; the lead
  // publishes the CTA's vote, waits for the grid's, and takes the ticket only
  // if the step runs.  Warps other than the lead never wait at the barrier.
  if (FUSED) {
    wait_bar(&bar_g[warp]);
    bool bad = false;
    for (int j = lane * 4; j < wn; j += 128) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        bad |= (__float_as_uint(grad_from_smem<GT>(sG, j + q)) & 0x7F800000u) == 0x7F800000u;
    }
    for (int k = nvec + static_cast<int>(threadIdx.x); k < len; k += kSmallThreads)
      bad |= (__float_as_uint(Grad<GT>::load1(T.g, start + k)) & 0x7F800000u) == 0x7F800000u;
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) s_bad[warp] = bad ? 1 : 0;
  }
  if (warp != kLead) {
    __threadfence_block();
    asm volatile("bar.arrive 1, %0;" ::"n"(kSmallThreads) : "memory");
  } else {
    asm volatile("bar.sync 1, %0;" ::"n"(kSmallThreads) : "memory");
    if (lane == 0) {
      if (FUSED) {
        bool any = false;
        for (int w = 0; w < kSmallWarps; ++w) any |= s_bad[w] != 0;
        amp_arrive(a.scratch, launch, any);   // the result is awaited after the stores
      } else {
        take_ticket_with(sa, t, s_next);
      }
    }
    __syncwarp();
  }

  // update the slice in place, four elements per lane per pass.  The grads
  // travel on their own barrier: the plain variant waits for it here (the
  // fused one did so before its scan) -- landing first is likely, not
  // ordered, and only the completed phase makes the copy visible
  if (!FUSED) wait_bar(&bar_g[warp]);
  wait_bar(&bar_s[warp]);
  if (landed) {
    for (int j = lane * 4; j < wn; j += 128) {
      float p[4], g[4], m[4], v[4];
      if (MODE == ADAMW_MODE_FP32) {
        const float4 x = *reinterpret_cast<const float4*>(sP + j * 4);
        p[0] = x.x; p[1] = x.y; p[2] = x.z; p[3] = x.w;
      } else {
        const uint2 h = *reinterpret_cast<const uint2*>(sP + j * 2);
        const uint2 r = *reinterpret_cast<const uint2*>(sR + j * 2);
        p[0] = rem_join(h.x & 0xFFFFu, r.x & 0xFFFFu);
        p[1] = rem_join(h.x >> 16, r.x >> 16);
        p[2] = rem_join(h.y & 0xFFFFu, r.y & 0xFFFFu);
        p[3] = rem_join(h.y >> 16, r.y >> 16);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) g[q] = grad_from_smem<GT>(sG, j + q);
      const float4 mm = *reinterpret_cast<const float4*>(sM + j * 4);
      const float4 vv = *reinterpret_cast<const float4*>(sV + j * 4);
      m[0] = mm.x; m[1] = mm.y; m[2] = mm.z; m[3] = mm.w;
      v[0] = vv.x; v[1] = vv.y; v[2] = vv.z; v[3] = vv.w;
#pragma unroll
      for (int q = 0; q < 4; ++q) update(p[q], g[q], m[q], v[q], s, decay);
      if (MODE == ADAMW_MODE_FP32) {
        *reinterpret_cast<float4*>(oP + j * 4) = make_float4(p[0], p[1], p[2], p[3]);
      } else {
        uint32_t h0, r0, h1, r1, h2, r2, h3, r3;
        rem_split(p[0], h0, r0);
        rem_split(p[1], h1, r1);
        rem_split(p[2], h2, r2);
        rem_split(p[3], h3, r3);
        *reinterpret_cast<uint2*>(oP + j * 2) = make_uint2(h0 | (h1 << 16), h2 | (h3 << 16));
        *reinterpret_cast<uint2*>(oR + j * 2) = make_uint2(r0 | (r1 << 16), r2 | (r3 << 16));
      }
      *reinterpret_cast<float4*>(oM + j * 4) = make_float4(m[0], m[1], m[2], m[3]);
      *reinterpret_cast<float4*>(oV + j * 4) = make_float4(v[0], v[1], v[2], v[3]);
    }
  }
  // the shared-memory results must be visible to the bulk copies that read them
  fence_proxy_async_smem();
  __syncwarp();

  // The stores go out at once, in the fused variant too: a skipped step is
  // rare, so its stores do not wait for the grid's vote -- a skip writes the
  // staged originals back once the first stores have completed.
  if (lane == 0 && wn > 0 && landed) {
    bulk_s2g(static_cast<unsigned char*>(T.p) + e0 * L::kP, oP, wn * L::kP);
    if (MODE == ADAMW_MODE_BF16_REM) bulk_s2g(T.rem + e0, oR, wn * 2);
    bulk_s2g(T.m + e0, oM, wn * 4);
    bulk_s2g(T.v + e0, oV, wn * 4);
    bulk_commit();
  }
  // the elements outside the bulk slices: a ragged tail (< 8), or the whole
  // piece of a tensor whose pointers are not 16-byte aligned (the fused
  // variant keeps each one's old values to write back on a skip)
  const TensorDesc td = as_desc(T);
  float old_p = 0.0f, old_m = 0.0f, old_v = 0.0f;
  uint16_t old_h = 0;
  int16_t old_r = 0;
  const int k_tail = nvec + static_cast<int>(threadIdx.x);
  // one element per thread of the CTA at most in the fused variant (the host
  // sends a plan whose pieces are not all 16-byte aligned to the other path)
  for (int k = k_tail; k < len; k += kSmallThreads) {
    if (FUSED) {
      if (MODE == ADAMW_MODE_FP32) {
        old_p = static_cast<const float*>(T.p)[start + k];
      } else {
        old_h = static_cast<const uint16_t*>(T.p)[start + k];
        old_r = T.rem[start + k];
      }
      old_m = T.m[start + k];
      old_v = T.v[start + k];
    }
    update_scalar<MODE, GT>(td, start + k, 1, s, decay);
  }
  if (FUSED) {
    // the grid's vote: the lead waits for it (bounded, 2 s) and takes the
    // CTA's ticket if the step stands; the other warps read it from the lead
    // (bounded too: a lead that never reports leaves the step as it stands,
    // fault bit 32)
    if (warp == kLead) {
      if (lane == 0) {
        const int v = amp_await(a.scratch, launch, found_inf_out);
        if (v == 0) take_ticket_with(sa, t, s_next);
        *static_cast<volatile int*>(&s_vote) = v;
      }
      __syncwarp();
    }
    int vote = *static_cast<volatile int*>(&s_vote);
    if (vote < 0) {
      const uint64_t t0 = global_ns();
      while ((vote = *static_cast<volatile int*>(&s_vote)) < 0) {
        __nanosleep(64);
        if (global_ns() - t0 > kWaitLimitNs) {
          if (lane == 0) atomicOr(&a.scratch->fault, 32u);
          vote = 2;
          break;
        }
      }
    }
    if (vote == 1) {   // skipped: the originals go back
      if (lane == 0 && wn > 0 && landed) {
        bulk_wait_all();   // the first stores have landed before the second ones start
        bulk_s2g(static_cast<unsigned char*>(T.p) + e0 * L::kP, sP, wn * L::kP);
        if (MODE == ADAMW_MODE_BF16_REM) bulk_s2g(T.rem + e0, sR, wn * 2);
        bulk_s2g(T.m + e0, sM, wn * 4);
        bulk_s2g(T.v + e0, sV, wn * 4);
        bulk_commit();
      }
      if (k_tail < len) {
        if (MODE == ADAMW_MODE_FP32) {
          static_cast<float*>(T.p)[start + k_tail] = old_p;
        } else {
          static_cast<uint16_t*>(T.p)[start + k_tail] = old_h;
          T.rem[start + k_tail] = old_r;
        }
        T.m[start + k_tail] = old_m;
        T.v[start + k_tail] = old_v;
      }
    }
  }
  // the CTA's shared memory stays allocated until the bulk stores have read it
  if (lane == 0) bulk_wait_read_all();
}

template <adamw_mode MODE, typename GT, bool FUSED>
cudaError_t launch_one(const SmallArgs& a, int grid, int smem, float* out, cudaStream_t st) {
  if (!FUSED) {
    step_small_kernel<MODE, GT, false><<<grid, kSmallThreads, smem, st>>>(a, out);
    return cudaGetLastError();
  }
  SmallArgs args = a;
  void* params[] = {&args, &out};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(step_small_kernel<MODE, GT, true>),
                                     dim3(grid), dim3(kSmallThreads), params,
                                     static_cast<size_t>(smem), st);
}

template <adamw_mode MODE, typename GT>
cudaError_t prepare_one(int smem, int smem_fused) {
  cudaError_t e = cudaFuncSetAttribute(step_small_kernel<MODE, GT, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess || smem_fused <= 0) return e;
  return cudaFuncSetAttribute(step_small_kernel<MODE, GT, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem_fused);
}

template <typename GT>
cudaError_t launch_mode(adamw_mode mode, const SmallArgs& a, int grid, int smem, bool fused,
                        float* out, cudaStream_t st) {
  if (mode == ADAMW_MODE_FP32)
    return fused ? launch_one<ADAMW_MODE_FP32, GT, true>(a, grid, smem, out, st)
                 : launch_one<ADAMW_MODE_FP32, GT, false>(a, grid, smem, out, st);
  if (mode == ADAMW_MODE_BF16_REM)
    return fused ? launch_one<ADAMW_MODE_BF16_REM, GT, true>(a, grid, smem, out, st)
                 : launch_one<ADAMW_MODE_BF16_REM, GT, false>(a, grid, smem, out, st);
  return cudaErrorInvalidValue;
}

template <typename GT>
cudaError_t prepare_mode(adamw_mode mode, int smem, int smem_fused) {
  if (mode == ADAMW_MODE_FP32) return prepare_one<ADAMW_MODE_FP32, GT>(smem, smem_fused);
  if (mode == ADAMW_MODE_BF16_REM) return prepare_one<ADAMW_MODE_BF16_REM, GT>(smem, smem_fused);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t prepare_step_small(adamw_mode mode, adamw_dtype gdt, int smem_bytes,
                               int smem_fused_bytes) {
  switch (gdt) {
    case ADAMW_F32: return prepare_mode<float>(mode, smem_bytes, smem_fused_bytes);
    case ADAMW_F16: return prepare_mode<__half>(mode, smem_bytes, smem_fused_bytes);
    case ADAMW_BF16: return prepare_mode<__nv_bfloat16>(mode, smem_bytes, smem_fused_bytes);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_step_small(adamw_mode mode, adamw_dtype gdt, const SmallArgs& a, int grid,
                              int smem_bytes, bool fused, float* found_inf_out, cudaStream_t s) {
  switch (gdt) {
    case ADAMW_F32: return launch_mode<float>(mode, a, grid, smem_bytes, fused, found_inf_out, s);
    case ADAMW_F16: return launch_mode<__half>(mode, a, grid, smem_bytes, fused, found_inf_out, s);
    case ADAMW_BF16:
      return launch_mode<__nv_bfloat16>(mode, a, grid, smem_bytes, fused, found_inf_out, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace adamw
