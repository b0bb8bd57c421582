// q4_kernels.cu -- the AdamW step with 4-bit blockwise-quantised moments.
//
// The 8-bit blockwise 2-state step of "Fix decoupled weight decay ordering in
// the CUDA Adam/AdEMAMix kernels" (bitsandbytes PR #2040) with 4-bit codes:
// dequantise m and v, run the strict-fp32 AdamW element update on the
// unquantised values, then re-quantise m' and v' per block of 128 elements
// (one fp32 absmax per block and per moment; nearest code, ties to the lower
// code).  Two codes per byte, the even element in the low nibble.
//
// Layout of the work: as in the 8-bit kernel every lane owns 8 consecutive
// elements of a 256-element warp span, so one half-warp owns one 128-element
// block; its absmax is a maximum over float32 bit patterns (exact and
// order-free) taken by two warp-wide reductions, one per half (1.5% faster on
// GB300 than a 16-lane xor-shuffle tree).  The 8 codes of a lane are one
// 32-bit word.
#include "step_common.cuh"

namespace adamw {
namespace {

constexpr int kQ4Block = 128;
constexpr int kQ4Span = 2 * kQ4Block;       // one warp: two blocks
constexpr int kQ4MinBlocks = 4;             // resident CTAs per SM the registers target
static_assert(16 * kVec == kQ4Block, "a half-warp holds one block");
static_assert(kQBlock % kQ4Span == 0, "chunks start on whole warp spans");

// Maximum over this lane's half-warp: two warp-wide reductions, each fed by
// one half (the other half gives 0, below every absolute-value bit pattern it
// competes with), then each lane keeps its own half's result.
__device__ __forceinline__ uint32_t half_warp_max(uint32_t x) {
  const bool upper = (threadIdx.x & 16) != 0;
  const uint32_t lo = __reduce_max_sync(0xFFFFFFFFu, upper ? 0u : x);
  const uint32_t hi = __reduce_max_sync(0xFFFFFFFFu, upper ? x : 0u);
  return upper ? hi : lo;
}

__device__ __forceinline__ uint8_t* codes(void* p) { return static_cast<uint8_t*>(p); }

// Nearest code of a normalised second moment x on the 4-bit v map, value
// (k+1)/16 for code k.  Its thresholds are the exact midpoints (k + 1.5)/16,
// so with y = 16x (exact: a power-of-two scaling) the code is
// #{k in 0..14 : y > k + 1.5} = clamp(ceil(y - 1.5), 0, 15), ties to the
// lower code.  The fma rounds 16x - 1.5 once: exactly wherever the result
// is at or above -0.75, and a result below that stays below 0 whatever its
// rounding; x is never negative, and a NaN converts to 0: code 0, as the
// table search gives.
__device__ __forceinline__ uint32_t v4_code(float x) {
  const int c = __float2int_ru(__fmaf_rn(x, 16.0f, -1.5f));
  return static_cast<uint32_t>(min(max(c, 0), 15));
}

// Codes of the 8 second moments one lane owns (the map has no zero: an
// all-zero block stores code 0, which dequantises to 0 through its absmax).
__device__ __forceinline__ void quant_v4(const float (&x)[8], const BlockNorm& n,
                                         uint32_t (&q)[8]) {
  if (n.bits == 0u) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0u;
  } else if (n.scale == 1.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = v4_code(__fmul_rn(x[i], n.inv));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = v4_code(__fmul_rn(__fmul_rn(x[i], n.scale), n.inv));
  }
}

__device__ __forceinline__ uint32_t pack_nibbles(const uint32_t (&q)[8]) {
  uint32_t w = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) w |= q[i] << (4 * i);
  return w;
}

template <typename GT, int R, bool SCALED>
__global__ void __launch_bounds__(kThreads, kQ4MinBlocks) step_q4_kernel(const StepArgs a) {
  constexpr int kSc = SCALED ? 1 : 0;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  QTables& qt = *reinterpret_cast<QTables*>(smem_raw);
  __shared__ Scal s_sc;
  __shared__ int s_skip;
  int t = 0;
  if (threadIdx.x == 0) s_skip = prologue(a, s_sc, t);
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.qt);
    uint4* dst = reinterpret_cast<uint4*>(smem_raw);
    for (int i = threadIdx.x; i < static_cast<int>(sizeof(QTables) / 16); i += kThreads)
      dst[i] = src[i];
  }
  __syncthreads();
  if (s_skip) return;
  const Scal s = s_sc;
  if (threadIdx.x == 0) take_ticket(a, t);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int half = lane >> 4;
  const uint32_t zc_m = qt.zero_code[0];

  for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
    const Chunk ch = a.chunks[c];
    const TensorDesc td = a.tensors[ch.tensor];
    // the code and absmax pointers are read again where they are used (the
    // step's stores may alias the descriptor, so the compiler keeps no copy
    // live across the pass): fewer spills at 64 registers
    const TensorDesc* const tdp = a.tensors + ch.tensor;
    const float decay = __fsub_rn(1.0f, __fmul_rn(s.lr, td.wd));
    const bool vec = td.vec_ok != 0;
    float* const pf = static_cast<float*>(td.p);

    // warp w owns the two blocks starting at `wb` of every pass; `e` is even
    for (int wb = warp * kQ4Span; wb < ch.len; wb += kPass) {
      const int64_t blk = (ch.start + wb) / kQ4Block + half;
      const int off = wb + lane * kVec;
      const int64_t e = ch.start + off;
      float m[8], v[8];
      uint32_t q_m[8], q_v[8];
      if (vec && wb + kQ4Span <= ch.len) {
        float p[8], gr[8];
        const float am = tdp->am[blk], av = tdp->av[blk];
        ld8f(pf + e, p);
        Grad<GT>::load8(td.g, e, gr);
        const uint32_t wm = __ldcs(reinterpret_cast<const uint32_t*>(codes(tdp->m) + e / 2));
        const uint32_t wv = __ldcs(reinterpret_cast<const uint32_t*>(codes(tdp->v) + e / 2));
        uint32_t mx_m = 0u, mx_v = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          m[i] = __fmul_rn(qt.map[0].value[(wm >> (4 * i)) & 0xFu], am);
          v[i] = __fmul_rn(qt.map[1].value[(wv >> (4 * i)) & 0xFu], av);
          update<kSc>(p[i], gr[i], m[i], v[i], s, decay);
          mx_m = max(mx_m, __float_as_uint(m[i]) & 0x7FFFFFFFu);
          // v' is never negative and never -0 (its NaN is the canonical,
          // positive one): its bits need no sign mask
          mx_v = max(mx_v, __float_as_uint(v[i]));
        }
        st8f(pf + e, p);
        const BlockNorm nm = block_norm(half_warp_max(mx_m));
        quant8<R>(m, nm, qt.map[0], zc_m, q_m);
        __stcs(reinterpret_cast<uint32_t*>(codes(tdp->m) + e / 2), pack_nibbles(q_m));
        const BlockNorm nv = block_norm(half_warp_max(mx_v));
        quant_v4(v, nv, q_v);
        __stcs(reinterpret_cast<uint32_t*>(codes(tdp->v) + e / 2), pack_nibbles(q_v));
        if ((lane & 15) == 0) {
          tdp->am[blk] = __uint_as_float(nm.bits);
          tdp->av[blk] = __uint_as_float(nv.bits);
        }
      } else {
        // the tail of a tensor (a half-warp's block may be partial or empty),
        // or a misaligned tensor: element by element
        const int n = max(0, min(kVec, ch.len - off));
        const bool has_block = wb + half * kQ4Block < ch.len;
        const float am = has_block ? tdp->am[blk] : 0.0f;
        const float av = has_block ? tdp->av[blk] : 0.0f;
        uint32_t mx_m = 0u, mx_v = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          m[i] = v[i] = 0.0f;
          if (i < n) {
            const int sh = 4 * (i & 1);
            float pi = pf[e + i];
            m[i] = __fmul_rn(qt.map[0].value[(codes(tdp->m)[(e + i) / 2] >> sh) & 0xFu], am);
            v[i] = __fmul_rn(qt.map[1].value[(codes(tdp->v)[(e + i) / 2] >> sh) & 0xFu], av);
            update<kSc>(pi, Grad<GT>::load1(td.g, e + i), m[i], v[i], s, decay);
            pf[e + i] = pi;
            mx_m = max(mx_m, __float_as_uint(m[i]) & 0x7FFFFFFFu);
            mx_v = max(mx_v, __float_as_uint(v[i]) & 0x7FFFFFFFu);
          }
        }
        const BlockNorm nm = block_norm(half_warp_max(mx_m));
        const BlockNorm nv = block_norm(half_warp_max(mx_v));
        quant8<R>(m, nm, qt.map[0], zc_m, q_m);
        quant_v4(v, nv, q_v);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          if (i < n) {
            const bool pair = i + 1 < n;
            codes(tdp->m)[(e + i) / 2] = static_cast<uint8_t>(q_m[i] | (pair ? q_m[i + 1] << 4 : 0u));
            codes(tdp->v)[(e + i) / 2] = static_cast<uint8_t>(q_v[i] | (pair ? q_v[i + 1] << 4 : 0u));
          }
        }
        if ((lane & 15) == 0 && has_block) {
          tdp->am[blk] = __uint_as_float(nm.bits);
          tdp->av[blk] = __uint_as_float(nv.bits);
        }
      }
    }
  }
}

template <typename GT, bool SCALED>
cudaError_t launch_q4_scaled(const StepArgs& a, int grid, cudaStream_t st) {
  if (a.refine <= 1)
    step_q4_kernel<GT, 1, SCALED><<<grid, kThreads, sizeof(QTables), st>>>(a);
  else if (a.refine <= 2)
    step_q4_kernel<GT, 2, SCALED><<<grid, kThreads, sizeof(QTables), st>>>(a);
  else
    step_q4_kernel<GT, kMaxRefine, SCALED><<<grid, kThreads, sizeof(QTables), st>>>(a);
  return cudaGetLastError();
}

template <typename GT>
cudaError_t launch_q4(const StepArgs& a, int grid, cudaStream_t st) {
  return a.grad_scale != nullptr ? launch_q4_scaled<GT, true>(a, grid, st)
                                 : launch_q4_scaled<GT, false>(a, grid, st);
}

}  // namespace

cudaError_t launch_step_q4(adamw_dtype gdt, const StepArgs& a, int grid, cudaStream_t s) {
  switch (gdt) {
    case ADAMW_F32: return launch_q4<float>(a, grid, s);
    case ADAMW_F16: return launch_q4<__half>(a, grid, s);
    case ADAMW_BF16: return launch_q4<__nv_bfloat16>(a, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t q4_occupancy(adamw_dtype gdt, int* bps, int* smem) {
  *smem = static_cast<int>(sizeof(QTables));
  switch (gdt) {
    case ADAMW_F32:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, step_q4_kernel<float, kMaxRefine, false>,
                                                           kThreads, *smem);
    case ADAMW_F16:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, step_q4_kernel<__half, kMaxRefine, false>,
                                                           kThreads, *smem);
    case ADAMW_BF16:
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          bps, step_q4_kernel<__nv_bfloat16, kMaxRefine, false>, kThreads, *smem);
  }
  return cudaErrorInvalidValue;
}

}  // namespace adamw
