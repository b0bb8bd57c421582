// step_kernels.cu -- the register-load step kernels for sm_103a: the 8-bit
// step and the fused non-finite check + step of adamw_step_amp for plans
// between the shared-memory-resident size and a few million elements.
//
// One persistent launch covers every tensor of a plan: CTAs stride over the
// plan's chunk table (up to 16384 contiguous elements of one tensor per chunk,
// a multiple of 256 but at a tensor's end), and each thread moves 8
// consecutive elements per pass with 128-bit streaming loads and stores.  The
// step is a pure HBM stream (28 B per element in fp32 mode, 26 in
// bf16+remainder mode, 14.06 in 8-bit mode), so there is no tensor-core work;
// the kernel's job is to keep enough bytes in flight.
//
// The element update is the decoupled-decay AdamW of "Fix decoupled weight
// decay ordering in the CUDA Adam/AdEMAMix kernels" (bitsandbytes PR #2040):
// decay and update both read the previous p.  Every operation is an explicit
// round-to-nearest intrinsic, so the compiler cannot contract a multiply and
// an add into an FMA and the result is the float32 sequence the header
// documents, bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "step_common.cuh"
#include "lane_tables.cuh"

namespace adamw {
namespace {

// ---------------------------------------------------------------- fp32 / bf16+rem
// The 8 consecutive elements one thread owns in one pass, in registers.
struct Group {
  float p[8], g[8], m[8], v[8];
};

template <adamw_mode MODE, typename GT>
__device__ __forceinline__ void load_group(const TensorDesc& td, int64_t e, Group& x) {
  if (MODE == ADAMW_MODE_FP32) {
    ld8f(static_cast<const float*>(td.p) + e, x.p);
  } else {
    uint32_t hw[4], rw[4];
    ld8u16(static_cast<const uint16_t*>(td.p) + e, hw);
    ld8u16(td.rem + e, rw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x.p[2 * i] = rem_join(hw[i] & 0xFFFFu, rw[i] & 0xFFFFu);
      x.p[2 * i + 1] = rem_join(hw[i] >> 16, rw[i] >> 16);
    }
  }
  Grad<GT>::load8(td.g, e, x.g);
  ld8f(static_cast<const float*>(td.m) + e, x.m);
  ld8f(static_cast<const float*>(td.v) + e, x.v);
}

template <adamw_mode MODE>
__device__ __forceinline__ void update_store_group(const TensorDesc& td, int64_t e, Group& x,
                                                   const Scal& s, float decay) {
#pragma unroll
  for (int i = 0; i < 8; ++i) update(x.p[i], x.g[i], x.m[i], x.v[i], s, decay);
  if (MODE == ADAMW_MODE_FP32) {
    st8f(static_cast<float*>(td.p) + e, x.p);
  } else {
    uint32_t hw[4], rw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h0, r0, h1, r1;
      rem_split(x.p[2 * i], h0, r0);
      rem_split(x.p[2 * i + 1], h1, r1);
      hw[i] = h0 | (h1 << 16);
      rw[i] = r0 | (r1 << 16);
    }
    st8u16(static_cast<uint16_t*>(td.p) + e, hw);
    st8u16(td.rem + e, rw);
  }
  st8f(static_cast<float*>(td.m) + e, x.m);
  st8f(static_cast<float*>(td.v) + e, x.v);
}

// A thread's position in its sequence of trips: chunk c (strided by the
// grid), element offset `base` inside it (strided by kPass * unroll).
struct Cursor {
  int64_t c;
  int base;
  Chunk ch;
};

// Move k to the next (chunk, offset) that holds work for this thread.
__device__ __forceinline__ bool seek(const StepArgs& a, Cursor& k) {
  while (k.c < a.n_chunks) {
    k.ch = a.chunks[k.c];
    if (k.base < k.ch.len) return true;
    k.c += gridDim.x;
    k.base = threadIdx.x * kVec;
  }
  return false;
}

template <adamw_mode MODE, typename GT, int U>
__device__ __forceinline__ void load_trip(const TensorDesc& td, const Cursor& k, bool vec,
                                          Group (&x)[U]) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int off = k.base + u * kPass;
    if (vec && off + kVec <= k.ch.len) load_group<MODE, GT>(td, k.ch.start + off, x[u]);
  }
}

// ---------------------------------------------------------------- fused AMP step
// Non-finite check and update in one cooperative launch: every CTA scans the
// grads of the chunks it will update, publishes whether it saw +-inf or NaN,
// and waits (bounded, 2 s) at a grid barrier; then all CTAs skip or update
// together.  For plans whose grads stay in L2 between the two passes.
template <typename GT>
__device__ __forceinline__ bool nonfinite1(const void* g, int64_t k) {
  if (sizeof(GT) == 4)
    return (static_cast<const uint32_t*>(g)[k] & 0x7F800000u) == 0x7F800000u;
  const uint32_t e = std::is_same<GT, __half>::value ? 0x7C00u : 0x7F80u;
  return (static_cast<const uint16_t*>(g)[k] & e) == e;
}

template <typename GT>
__device__ __forceinline__ bool nonfinite8(const void* g, int64_t e) {
  float x[8];
  Grad<GT>::load8(g, e, x);
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) bad |= (__float_as_uint(x[i]) & 0x7F800000u) == 0x7F800000u;
  return bad;
}

template <adamw_mode MODE, typename GT>
__global__ void __launch_bounds__(kThreads, Tune<MODE>::min_blocks)
step_fused_amp_kernel(const StepArgs a, float* found_inf_out) {
  constexpr int kUnroll = Tune<MODE>::unroll;
  __shared__ Scal s_sc;
  __shared__ int s_skip;
  StepScratch* const sc = a.scratch;

  // 1. scan this CTA's grads (the same elements it updates below)
  bool bad = false;
  for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
    const Chunk ch = a.chunks[c];
    const TensorDesc& td = a.tensors[ch.tensor];
    for (int off = threadIdx.x * kVec; off < ch.len; off += kPass) {
      if (td.vec_ok && off + kVec <= ch.len) {
        bad |= nonfinite8<GT>(td.g, ch.start + off);
      } else {
        const int n = min(kVec, ch.len - off);
        for (int i = 0; i < n; ++i) bad |= nonfinite1<GT>(td.g, ch.start + off + i);
      }
    }
  }
  bad = __syncthreads_or(bad);

  // 2. grid barrier: publish, then wait until every CTA of this launch has
  if (threadIdx.x == 0) s_skip = amp_grid_vote(sc, bad, found_inf_out);
  __syncthreads();
  if (s_skip) return;

  // 3. the step itself, loads into registers
  int t = 0;
  if (threadIdx.x == 0) s_skip = prologue(a, s_sc, t);
  __syncthreads();
  const Scal s = s_sc;
  if (threadIdx.x == 0) take_ticket(a, t);
  Cursor k{static_cast<int64_t>(blockIdx.x), static_cast<int>(threadIdx.x) * kVec, Chunk{}};
  bool have = seek(a, k);
  while (have) {
    const TensorDesc td = a.tensors[k.ch.tensor];
    const float decay = __fsub_rn(1.0f, __fmul_rn(s.lr, td.wd));
    const bool vec = td.vec_ok != 0;
    Group x[kUnroll];
    load_trip<MODE, GT, kUnroll>(td, k, vec, x);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int off = k.base + u * kPass;
      if (vec && off + kVec <= k.ch.len)
        update_store_group<MODE>(td, k.ch.start + off, x[u], s, decay);
      else if (off < k.ch.len)
        update_scalar<MODE, GT>(td, k.ch.start + off, min(kVec, k.ch.len - off), s, decay);
    }
    k.base += kPass * kUnroll;
    if (k.base >= k.ch.len) {
      k.c += gridDim.x;
      k.base = threadIdx.x * kVec;
      have = seek(a, k);
    }
  }
}

template <typename GT>
cudaError_t launch_fused_mode(adamw_mode mode, const StepArgs& a, int grid, float* out,
                              cudaStream_t st) {
  StepArgs args = a;
  void* params[] = {&args, &out};
  if (mode == ADAMW_MODE_FP32)
    return cudaLaunchCooperativeKernel(
        reinterpret_cast<const void*>(step_fused_amp_kernel<ADAMW_MODE_FP32, GT>), dim3(grid),
        dim3(kThreads), params, 0, st);
  if (mode == ADAMW_MODE_BF16_REM)
    return cudaLaunchCooperativeKernel(
        reinterpret_cast<const void*>(step_fused_amp_kernel<ADAMW_MODE_BF16_REM, GT>), dim3(grid),
        dim3(kThreads), params, 0, st);
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- 8-bit states
// One CTA of kQ8Threads per SM; every warp owns one 256-element block per
// pass, each lane 8 consecutive elements.  The code tables are lane-private
// copies in shared memory (lane_tables.cuh).
constexpr int kQ8Smem = static_cast<int>(sizeof(LaneTables<256>));

__device__ __forceinline__ uint8_t* codes_m(const TensorDesc* td) {
  return static_cast<uint8_t*>(td->m);
}
__device__ __forceinline__ uint8_t* codes_v(const TensorDesc* td) {
  return static_cast<uint8_t*>(td->v);
}

template <typename GT, int R, bool SCALED>
__global__ void __launch_bounds__(kQ8Threads, 1) step_q8_kernel(const StepArgs a) {
  constexpr int kSc = SCALED ? 1 : 0;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  LaneTables<256>& lt = *reinterpret_cast<LaneTables<256>*>(smem_raw);
  __shared__ Scal s_sc;
  __shared__ int s_skip;
  int t = 0;
  if (threadIdx.x == 0) s_skip = prologue(a, s_sc, t);
  fill_lane_tables<256>(lt, a.qt);
  __syncthreads();
  if (s_skip) return;
  const Scal s = s_sc;
  if (threadIdx.x == 0) take_ticket(a, t);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const uint32_t zc_m = a.qt->zero_code[0], zc_v = a.qt->zero_code[1];

  for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
    const Chunk ch = a.chunks[c];
    const TensorDesc td = a.tensors[ch.tensor];
    // the code and absmax pointers are read again where they are used (the
    // step's stores may alias the descriptor, so the compiler keeps no copy
    // live across the pass): no spills at 64 registers
    const TensorDesc* const tdp = a.tensors + ch.tensor;
    const float decay = __fsub_rn(1.0f, __fmul_rn(s.lr, td.wd));
    const bool vec = td.vec_ok != 0;
    float* const pf = static_cast<float*>(td.p);

    // warp w owns the 256-element block starting at `wb` of every pass
    for (int wb = warp * kQBlock; wb < ch.len; wb += kQ8Pass) {
      const int64_t blk = (ch.start + wb) / kQBlock;   // block-aligned within the tensor
      const int off = wb + lane * kVec;
      const int64_t e = ch.start + off;
      const float am = tdp->am[blk], av = tdp->av[blk];
      float p[8], gr[8], m[8], v[8];
      uint32_t q_m[8], q_v[8];
      // a whole block on the 128-bit path: no per-element predicates
      if (vec && wb + kQBlock <= ch.len) {
        ld8f(pf + e, p);
        Grad<GT>::load8(td.g, e, gr);
        const uint2 qm = __ldcs(reinterpret_cast<const uint2*>(codes_m(tdp) + e));
        const uint2 qv = __ldcs(reinterpret_cast<const uint2*>(codes_v(tdp) + e));
        uint32_t mx_m = 0u, mx_v = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t wm = i < 4 ? qm.x : qm.y, wv = i < 4 ? qv.x : qv.y;
          const int sh = (i & 3) * 8;
          m[i] = __fmul_rn(lt.value[0][(wm >> sh) & 0xFFu][lane], am);
          v[i] = __fmul_rn(lt.value[1][(wv >> sh) & 0xFFu][lane], av);
          update<kSc>(p[i], gr[i], m[i], v[i], s, decay);
          mx_m = max(mx_m, __float_as_uint(m[i]) & 0x7FFFFFFFu);
          // v' = b2*v + (1-b2)*g*g is never negative and never -0 (its NaN
          // is the canonical, positive one): its bits need no sign mask
          mx_v = max(mx_v, __float_as_uint(v[i]));
        }
        // store each result as soon as it is final: short live ranges keep the
        // kernel within its 64 registers
        st8f(pf + e, p);
        const BlockNorm nm = block_norm(__reduce_max_sync(0xFFFFFFFFu, mx_m));
        lane_quant8<256, 0, R>(lt, m, nm, zc_m, lane, q_m);
        __stcs(reinterpret_cast<uint2*>(codes_m(tdp) + e), pack8(q_m));
        const BlockNorm nv = block_norm(__reduce_max_sync(0xFFFFFFFFu, mx_v));
        lane_quant8<256, 1, R>(lt, v, nv, zc_v, lane, q_v);
        __stcs(reinterpret_cast<uint2*>(codes_v(tdp) + e), pack8(q_v));
        if (lane == 0) {
          tdp->am[blk] = __uint_as_float(nm.bits);
          tdp->av[blk] = __uint_as_float(nv.bits);
        }
      } else {
        // the last (partial) block of a tensor, or a misaligned tensor
        const int n = max(0, min(kVec, ch.len - off));
        uint32_t mx_m = 0u, mx_v = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          p[i] = gr[i] = m[i] = v[i] = 0.0f;
          if (i < n) {
            p[i] = pf[e + i];
            gr[i] = Grad<GT>::load1(td.g, e + i);
            m[i] = __fmul_rn(lt.value[0][codes_m(tdp)[e + i]][lane], am);
            v[i] = __fmul_rn(lt.value[1][codes_v(tdp)[e + i]][lane], av);
            update<kSc>(p[i], gr[i], m[i], v[i], s, decay);
            mx_m = max(mx_m, __float_as_uint(m[i]) & 0x7FFFFFFFu);
            mx_v = max(mx_v, __float_as_uint(v[i]) & 0x7FFFFFFFu);
          }
        }
        const BlockNorm nm = block_norm(__reduce_max_sync(0xFFFFFFFFu, mx_m));
        const BlockNorm nv = block_norm(__reduce_max_sync(0xFFFFFFFFu, mx_v));
        lane_quant8<256, 0, R>(lt, m, nm, zc_m, lane, q_m);
        lane_quant8<256, 1, R>(lt, v, nv, zc_v, lane, q_v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < n) {
            pf[e + i] = p[i];
            codes_m(tdp)[e + i] = static_cast<uint8_t>(q_m[i]);
            codes_v(tdp)[e + i] = static_cast<uint8_t>(q_v[i]);
          }
        }
        if (lane == 0) {
          tdp->am[blk] = __uint_as_float(nm.bits);
          tdp->av[blk] = __uint_as_float(nv.bits);
        }
      }
    }
  }
}

template <typename GT, bool SCALED>
cudaError_t launch_q8(const StepArgs& a, int grid, cudaStream_t st) {
  if (a.refine <= 1)
    step_q8_kernel<GT, 1, SCALED><<<grid, kQ8Threads, kQ8Smem, st>>>(a);
  else if (a.refine <= 2)
    step_q8_kernel<GT, 2, SCALED><<<grid, kQ8Threads, kQ8Smem, st>>>(a);
  else
    step_q8_kernel<GT, kMaxRefine, SCALED><<<grid, kQ8Threads, kQ8Smem, st>>>(a);
  return cudaGetLastError();
}

template <typename GT, bool SCALED>
cudaError_t q8_smem_limits() {
  cudaError_t e = cudaFuncSetAttribute(step_q8_kernel<GT, 1, SCALED>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kQ8Smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(step_q8_kernel<GT, 2, SCALED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kQ8Smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(step_q8_kernel<GT, kMaxRefine, SCALED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kQ8Smem);
  return e;
}

template <typename GT>
cudaError_t launch_mode(adamw_mode mode, const StepArgs& a, int grid, cudaStream_t st) {
  switch (mode) {
    case ADAMW_MODE_Q8:
      if (a.grad_scale != nullptr) return launch_q8<GT, true>(a, grid, st);
      return launch_q8<GT, false>(a, grid, st);
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename GT>
cudaError_t occupancy_mode(adamw_mode mode, int* bps, int* smem) {
  switch (mode) {
    case ADAMW_MODE_Q8: {
      // the lane-private tables exceed the 48 KB default: raise the limit of
      // each variant (before any launch), then ask for the occupancy
      *smem = kQ8Smem;
      cudaError_t e = q8_smem_limits<GT, false>();
      if (e == cudaSuccess) e = q8_smem_limits<GT, true>();
      if (e != cudaSuccess) return e;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          bps, step_q8_kernel<GT, kMaxRefine, false>, kQ8Threads, kQ8Smem);
    }
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

template <typename GT>
cudaError_t fused_occ_mode(adamw_mode mode, int* bps) {
  if (mode == ADAMW_MODE_FP32)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        bps, step_fused_amp_kernel<ADAMW_MODE_FP32, GT>, kThreads, 0);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      bps, step_fused_amp_kernel<ADAMW_MODE_BF16_REM, GT>, kThreads, 0);
}

cudaError_t fused_occupancy(adamw_mode mode, adamw_dtype gdt, int* bps) {
  switch (gdt) {
    case ADAMW_F32: return fused_occ_mode<float>(mode, bps);
    case ADAMW_F16: return fused_occ_mode<__half>(mode, bps);
    case ADAMW_BF16: return fused_occ_mode<__nv_bfloat16>(mode, bps);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_step_fused_amp(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                                  float* found_inf_out, cudaStream_t s) {
  switch (gdt) {
    case ADAMW_F32: return launch_fused_mode<float>(mode, a, grid, found_inf_out, s);
    case ADAMW_F16: return launch_fused_mode<__half>(mode, a, grid, found_inf_out, s);
    case ADAMW_BF16: return launch_fused_mode<__nv_bfloat16>(mode, a, grid, found_inf_out, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_step(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                        cudaStream_t s) {
  switch (gdt) {
    case ADAMW_F32: return launch_mode<float>(mode, a, grid, s);
    case ADAMW_F16: return launch_mode<__half>(mode, a, grid, s);
    case ADAMW_BF16: return launch_mode<__nv_bfloat16>(mode, a, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t step_occupancy(adamw_mode mode, adamw_dtype gdt, int* bps, int* smem) {
  switch (gdt) {
    case ADAMW_F32: return occupancy_mode<float>(mode, bps, smem);
    case ADAMW_F16: return occupancy_mode<__half>(mode, bps, smem);
    case ADAMW_BF16: return occupancy_mode<__nv_bfloat16>(mode, bps, smem);
  }
  return cudaErrorInvalidValue;
}

}  // namespace adamw
