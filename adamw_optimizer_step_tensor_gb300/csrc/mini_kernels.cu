// mini_kernels.cu -- the block reduction of the Adam-mini step.
//
// "Adam-mini <> DTensor", AdamWMini listing: a head or a whole tensor shares
// one second moment, v = b2*v + (1-b2)*mean(g*g) over the block, and every
// element of the block then moves by lr * m' * ((1/bc1) / h) with
// h = sqrt(v)/sqrt(bc2) + eps.  This kernel computes, for every block longer
// than one element, the mean of g*g, the new v and r = fl(1/bc1) / h; the
// element update is the bulk-staged step kernel (kAlgoMini), launched next on
// the same stream.
//
// Chunks never straddle blocks.  Each warp sums g*g over one chunk on its
// own -- no CTA barrier inside the walk, so a warp whose loads are back never
// waits for the others -- with kRedLoads loads of 8 grads per lane in flight.
// Each lane sums the 32 squares of one round of loads as an unevaluated pair
// of float32 (s, c): each square split exactly into x*x = p + e with one fma,
// each addition into s made error-free with TwoSum, the errors gathered in c
// (Ogita, Rump and Oishi, "Accurate sum and dot product", 2005: relative error
// about (32*2^-24)^2, with no float64 operation per element, which GB300 runs
// at a small fraction of its float32 rate), and adds s + c to its float64
// total; a round whose pair is not finite is summed again with float64
// squares.  The lanes' totals meet in a fixed float64 xor tree.  A block of one
// chunk is finalised by that warp; otherwise the warp whose arrival completes
// the block's count adds the block's chunk sums (float64, each lane a fixed
// stride of them, then a fixed xor tree), finalises the block and clears the
// count for the next step.  Nothing waits on another warp.
#include "step_common.cuh"

namespace adamw {
namespace {

constexpr int kRedThreads = kRedWarps * 32;
constexpr float kF32Max = 3.40282347e38f;   // the largest finite float32
constexpr int kRedLoads = 4;   // 8-grad loads in flight per lane

// (s, c) += x*x: TwoProduct of the square by fma, TwoSum of the addition.
// EXACT_SQUARE: x has at most 12 significant bits (an unscaled 16-bit grad),
// so x*x is exact in float32 wherever it is a normal number and the product's
// error term is 0: it is not computed.
template <bool EXACT_SQUARE>
__device__ __forceinline__ void add_square(float& s, float& c, float x) {
  const float p = __fmul_rn(x, x);
  const float t = __fadd_rn(s, p);
  const float bp = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp));
  s = t;
  if constexpr (EXACT_SQUARE) {
    c = __fadd_rn(c, err);
  } else {
    const float e = __fmaf_rn(x, x, -p);
    c = __fadd_rn(c, __fadd_rn(err, e));
  }
}

// 8 consecutive raw grads of one lane, kept as loaded (16-bit grads stay
// packed until they are squared).
template <typename GT>
struct RawGrads {
  uint4 w[sizeof(GT) == 4 ? 2 : 1];
};

template <typename GT>
__device__ __forceinline__ void load_raw(const void* g, int64_t e, int n, bool vec,
                                         RawGrads<GT>& r) {
  if (vec && n == kVec) {
    const uint4* q = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(g) +
                                                    e * static_cast<int64_t>(sizeof(GT)));
    r.w[0] = __ldcs(q);
    if constexpr (sizeof(GT) == 4) r.w[1] = __ldcs(q + 1);
  } else {
    uint32_t b[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      b[q] = 0u;   // +0 in every grad type: its square adds nothing
      if (q < n) {
        if constexpr (sizeof(GT) == 4)
          b[q] = static_cast<const uint32_t*>(g)[e + q];
        else
          b[q] = static_cast<const uint16_t*>(g)[e + q];
      }
    }
    if constexpr (sizeof(GT) == 4) {
      r.w[0] = make_uint4(b[0], b[1], b[2], b[3]);
      r.w[1] = make_uint4(b[4], b[5], b[6], b[7]);
    } else {
      r.w[0] = make_uint4(b[0] | b[1] << 16, b[2] | b[3] << 16, b[4] | b[5] << 16,
                          b[6] | b[7] << 16);
    }
  }
}

// Grad q (0..7) of a group, widened exactly to float32.
template <typename GT>
__device__ __forceinline__ float raw_grad(const RawGrads<GT>& r, int q) {
  if constexpr (sizeof(GT) == 4) {
    const uint4 w = r.w[q >> 2];
    const uint32_t x = (q & 3) == 0 ? w.x : (q & 3) == 1 ? w.y : (q & 3) == 2 ? w.z : w.w;
    return __uint_as_float(x);
  } else {
    const uint4 w = r.w[0];
    const uint32_t x = (q >> 1) == 0 ? w.x : (q >> 1) == 1 ? w.y : (q >> 1) == 2 ? w.z : w.w;
    const uint32_t h = (q & 1) ? x >> 16 : x & 0xFFFFu;
    if constexpr (std::is_same<GT, __half>::value) return f16_to_f32(h);
    return bf16_to_f32(h);
  }
}

// v, h and r of one block from the float64 sum of g*g over it.
__device__ void finalise(const StepArgs& a, const MiniArgs& ma, int32_t b, double sum,
                         const Scal& s) {
  const MiniBlock blk = ma.blocks[b];
  float* const v = static_cast<float*>(a.tensors[blk.tensor].v) + blk.v_index;
  const float mean = __double2float_rn(__ddiv_rn(sum, static_cast<double>(blk.len)));
  const float v1 = __fadd_rn(__fmul_rn(s.b2, *v), __fmul_rn(s.omb2, mean));
  *v = v1;
  const float h = __fadd_rn(__fmul_rn(__fsqrt_rn(v1), s.inv_sqrt_bc2), s.eps);
  ma.blk_r[b] = __fdiv_rn(s.rbc1, h);
}

// SCALED: the launch has a loss scale (the unscale is then applied to every
// grad; x * 1 is exact, so a scale of 1 changes nothing) -- a template
// parameter, so the unscaled step spends no instruction per element on it.
template <typename GT, bool SCALED>
__global__ void __launch_bounds__(kRedThreads, sizeof(GT) == 4 ? 4 : 5) mini_reduce_kernel(const StepArgs a,
                                                                  const MiniArgs ma) {
  __shared__ Scal s_sc;
  __shared__ int s_skip;
  int t = 0;
  if (threadIdx.x == 0) s_skip = prologue(a, s_sc, t);
  __syncthreads();
  if (s_skip) return;
  const Scal s = s_sc;
  const int lane = threadIdx.x & 31;
  constexpr int kStride = 32 * kVec;   // elements between one lane's groups
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * kRedWarps;
  // bf16 (8 significant bits) and fp16 (11) squares are exact in float32
  constexpr bool kExactSquare = !SCALED && sizeof(GT) == 2;

  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kRedWarps + (threadIdx.x >> 5); i < ma.n_red;
       i += n_warps) {
    const int64_t c = ma.red_chunks[i];
    const Chunk ch = a.chunks[c];
    const TensorDesc* const tdp = a.tensors + ch.tensor;
    const void* const g = tdp->g;
    const bool vec = tdp->vec_ok != 0;
    // lane l takes the groups of 8 at l*8, l*8 + 256, ...: each load of the
    // warp covers 256 consecutive grads; the squares go in in element order,
    // 8 * kRedLoads into one float32 pair, which then joins the lane's float64
    // total (so no pair takes more than 32 squares)
    double lane_sum = 0.0;
    for (int off0 = lane * kVec; off0 < ch.len; off0 += kRedLoads * kStride) {
      RawGrads<GT> r[kRedLoads];
#pragma unroll
      for (int u = 0; u < kRedLoads; ++u) {
        const int off = off0 + u * kStride;
        load_raw<GT>(g, ch.start + off, max(0, min(kVec, ch.len - off)), vec, r[u]);
      }
      float sum = 0.0f, comp = 0.0f;
#pragma unroll
      for (int u = 0; u < kRedLoads; ++u) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float x = raw_grad<GT>(r[u], q);
          add_square<kExactSquare>(sum, comp, SCALED ? __fmul_rn(x, s.inv_scale) : x);
        }
      }
      if (fabsf(sum) <= kF32Max) {
        lane_sum += static_cast<double>(sum) + static_cast<double>(comp);
      } else {
        // a NaN or infinite grad, or a square or partial sum past the float32
        // range, where the split of a square is not exact (inf - inf): this
        // round again with float64 squares, exact for every float32 -- inf
        // and NaN as the definition gives them, and a finite mean where the
        // float64 sum of squares allows one
        // (the grads are loaded again: this rare path keeps no registers
        // live through the common one)
        double acc = 0.0;
#pragma unroll
        for (int u = 0; u < kRedLoads; ++u) {
          const int off = off0 + u * kStride;
          RawGrads<GT> again;
          load_raw<GT>(g, ch.start + off, max(0, min(kVec, ch.len - off)), vec, again);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float x = raw_grad<GT>(again, q);
            const double xd = static_cast<double>(SCALED ? __fmul_rn(x, s.inv_scale) : x);
            acc += xd * xd;
          }
        }
        lane_sum += acc;
      }
    }
    // the lanes' totals in a fixed xor tree (float64 addition commutes: every
    // lane ends with the same chunk sum)
    double d = lane_sum;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
    const int32_t b = a.chunk_blk[c];
    const MiniBlock blk = ma.blocks[b];
    if (blk.n_chunks == 1) {
      if (lane == 0) finalise(a, ma, b, d, s);
      continue;
    }
    uint32_t last = 0u;
    if (lane == 0) {
      ma.partial[c] = d;
      __threadfence();
      last = atomicAdd(&ma.arrived[b], 1u) == static_cast<uint32_t>(blk.n_chunks - 1) ? 1u : 0u;
    }
    if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
      // this warp completed the block: add its chunk sums, each lane a fixed
      // stride of them, then the fixed xor tree
      __threadfence();
      double part = 0.0;
      for (int64_t k = lane; k < blk.n_chunks; k += 32)
        part += __ldcg(&ma.partial[blk.first_chunk + k]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
      if (lane == 0) {
        finalise(a, ma, b, part, s);
        ma.arrived[b] = 0u;
      }
    }
  }
}

template <typename GT>
cudaError_t launch_reduce(const StepArgs& a, const MiniArgs& ma, int grid, cudaStream_t s) {
  if (a.grad_scale != nullptr)
    mini_reduce_kernel<GT, true><<<grid, kRedThreads, 0, s>>>(a, ma);
  else
    mini_reduce_kernel<GT, false><<<grid, kRedThreads, 0, s>>>(a, ma);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mini_reduce(adamw_dtype gdt, const StepArgs& a, const MiniArgs& ma, int grid,
                               cudaStream_t s) {
  switch (gdt) {
    case ADAMW_F32: return launch_reduce<float>(a, ma, grid, s);
    case ADAMW_F16: return launch_reduce<__half>(a, ma, grid, s);
    case ADAMW_BF16: return launch_reduce<__nv_bfloat16>(a, ma, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace adamw
