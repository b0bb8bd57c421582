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
// Chunks never straddle blocks.  Each CTA sums g*g over one chunk: every
// thread keeps its sum as an unevaluated pair of float32 (s, c) -- each square
// split exactly into x*x = p + e with one fma, each addition into s made
// error-free with TwoSum, the errors gathered in c (Ogita, Rump and Oishi,
// "Accurate sum and dot product", 2005: relative error about (n*2^-24)^2 for
// the n = 64 squares of a thread, with no float64 operation per element,
// which GB300 runs at a small fraction of its float32 rate) -- the pairs are added in float64 in a fixed
// tree, and the chunk's sum is stored.  A block of one chunk is
// finalised by that CTA; otherwise the CTA that completes the block's arrival
// count adds the block's chunk sums (float64, each thread a fixed stride of
// them, then the fixed tree) and finalises it, then clears the count for the
// next step.  Nothing waits on another CTA.
#include "step_common.cuh"

namespace adamw {
namespace {

constexpr int kRedThreads = 256;

// (s, c) += x*x: TwoProduct of the square by fma, TwoSum of the addition.
__device__ __forceinline__ void add_square(float& s, float& c, float x) {
  const float p = __fmul_rn(x, x);
  const float e = __fmaf_rn(x, x, -p);
  const float t = __fadd_rn(s, p);
  const float bp = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp));
  s = t;
  c = __fadd_rn(c, __fadd_rn(err, e));
}

// (s, c) += (s2, c2) for two error-free pairs: TwoSum of the leading parts,
// the rounding error joins the trailing parts.
__device__ __forceinline__ void add_pair(float& s, float& c, float s2, float c2) {
  const float t = __fadd_rn(s, s2);
  const float bp = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(s2, bp));
  s = t;
  c = __fadd_rn(__fadd_rn(c, c2), err);
}

// The sum over the CTA of one pair per thread, in a fixed order (xor tree of
// pairs in each warp, then the warps' pairs in float64 in order).  The result
// is valid in thread 0.  Float64 work stays at 16 additions per CTA: GB300
// issues float64 at a small fraction of its float32 rate.
__device__ __forceinline__ double cta_pair_sum(float s, float c, float2* s_pair) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    add_pair(s, c, __shfl_xor_sync(0xFFFFFFFFu, s, o), __shfl_xor_sync(0xFFFFFFFFu, c, o));
  if ((threadIdx.x & 31) == 0) s_pair[threadIdx.x >> 5] = make_float2(s, c);
  __syncthreads();
  double total = 0.0;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < kRedThreads / 32; ++w) {
      total += static_cast<double>(s_pair[w].x);
      total += static_cast<double>(s_pair[w].y);
    }
  }
  __syncthreads();
  return total;
}

// The float64 sum of one value per thread, in a fixed order; valid in thread 0.
__device__ __forceinline__ double cta_sum(double x, double* s_warp) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = x;
  __syncthreads();
  double total = 0.0;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < kRedThreads / 32; ++w) total += s_warp[w];
  }
  __syncthreads();
  return total;
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

template <typename GT>
__global__ void __launch_bounds__(kRedThreads) mini_reduce_kernel(const StepArgs a,
                                                                  const MiniArgs ma) {
  __shared__ Scal s_sc;
  __shared__ int s_skip;
  __shared__ double s_warp[kRedThreads / 32];
  __shared__ float2 s_pair[kRedThreads / 32];
  __shared__ int s_last;
  int t = 0;
  if (threadIdx.x == 0) s_skip = prologue(a, s_sc, t);
  __syncthreads();
  if (s_skip) return;
  const Scal s = s_sc;

  for (int64_t i = blockIdx.x; i < ma.n_red; i += gridDim.x) {
    const int64_t c = ma.red_chunks[i];
    const Chunk ch = a.chunks[c];
    const TensorDesc td = a.tensors[ch.tensor];
    float sum = 0.0f, comp = 0.0f;
    for (int off = threadIdx.x * kVec; off < ch.len; off += kRedThreads * kVec) {
      const int64_t e = ch.start + off;
      float g[8];
      const int n = min(kVec, ch.len - off);
      if (td.vec_ok && n == kVec) {
        Grad<GT>::load8(td.g, e, g);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) g[q] = q < n ? Grad<GT>::load1(td.g, e + q) : 0.0f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float x = s.scaled ? __fmul_rn(g[q], s.inv_scale) : g[q];
        add_square(sum, comp, x);
      }
    }
    const double d = cta_pair_sum(sum, comp, s_pair);
    const int32_t b = a.chunk_blk[c];
    const MiniBlock blk = ma.blocks[b];
    if (blk.n_chunks == 1) {
      if (threadIdx.x == 0) finalise(a, ma, b, d, s);
    } else {
      if (threadIdx.x == 0) {
        ma.partial[c] = d;
        __threadfence();
        const uint32_t prev = atomicAdd(&ma.arrived[b], 1u);
        s_last = prev == static_cast<uint32_t>(blk.n_chunks - 1);
      }
      __syncthreads();
      if (s_last) {
        // this CTA completed the block: add its chunk sums, each thread a
        // fixed stride of them, then the fixed tree
        __threadfence();
        double part = 0.0;
        for (int64_t k = threadIdx.x; k < blk.n_chunks; k += kRedThreads)
          part += __ldcg(&ma.partial[blk.first_chunk + k]);
        const double total = cta_sum(part, s_warp);
        if (threadIdx.x == 0) {
          finalise(a, ma, b, total, s);
          ma.arrived[b] = 0u;
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_mini_reduce(adamw_dtype gdt, const StepArgs& a, const MiniArgs& ma, int grid,
                               cudaStream_t s) {
  switch (gdt) {
    case ADAMW_F32: mini_reduce_kernel<float><<<grid, kRedThreads, 0, s>>>(a, ma); break;
    case ADAMW_F16: mini_reduce_kernel<__half><<<grid, kRedThreads, 0, s>>>(a, ma); break;
    case ADAMW_BF16: mini_reduce_kernel<__nv_bfloat16><<<grid, kRedThreads, 0, s>>>(a, ma); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace adamw
