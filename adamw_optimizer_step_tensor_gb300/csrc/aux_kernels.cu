// aux_kernels.cu -- the non-finite grad check, the remainder split/join and
// the Q8 state export/import kernels.
#include "internal.h"
#include "step_common.cuh"

namespace adamw {
namespace {

// Exponent field all ones <=> +-inf or NaN.
template <adamw_dtype D> struct NonFinite;
template <> struct NonFinite<ADAMW_F32> {
  static __device__ __forceinline__ bool vec(const void* g, int64_t e) {
    const uint4* q = reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(g) + e);
    const uint4 a = __ldcs(q), b = __ldcs(q + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) bad |= (w[i] & 0x7F800000u) == 0x7F800000u;
    return bad;
  }
  static __device__ __forceinline__ bool one(const void* g, int64_t e) {
    return (static_cast<const uint32_t*>(g)[e] & 0x7F800000u) == 0x7F800000u;
  }
};
template <uint32_t kExp> struct NonFinite16 {
  static __device__ __forceinline__ bool vec(const void* g, int64_t e) {
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(g) + e));
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      bad |= ((w[i] & kExp) == kExp) || (((w[i] >> 16) & kExp) == kExp);
    return bad;
  }
  static __device__ __forceinline__ bool one(const void* g, int64_t e) {
    return (static_cast<const uint16_t*>(g)[e] & kExp) == kExp;
  }
};
template <> struct NonFinite<ADAMW_F16> : NonFinite16<0x7C00u> {};
template <> struct NonFinite<ADAMW_BF16> : NonFinite16<0x7F80u> {};

template <adamw_dtype D>
__global__ void __launch_bounds__(kThreads)
nonfinite_kernel(const TensorDesc* tensors, const Chunk* chunks, int64_t n_chunks,
                 float* found_inf) {
  bool bad = false;
  for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const TensorDesc& td = tensors[ch.tensor];
    const bool vec = td.vec_ok != 0;
    for (int off = threadIdx.x * kVec; off < ch.len; off += kPass) {
      const int64_t e = ch.start + off;
      if (vec && off + kVec <= ch.len) {
        bad |= NonFinite<D>::vec(td.g, e);
      } else {
        const int n = min(kVec, ch.len - off);
        for (int i = 0; i < n; ++i) bad |= NonFinite<D>::one(td.g, e + i);
      }
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) *found_inf = 1.0f;
}

__global__ void split_kernel(const float* __restrict__ master, uint16_t* __restrict__ hi,
                             int16_t* __restrict__ rem, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint32_t h, r;
    rem_split(master[i], h, r);
    hi[i] = static_cast<uint16_t>(h);
    rem[i] = static_cast<int16_t>(static_cast<uint16_t>(r));
  }
}

__global__ void join_kernel(const uint16_t* __restrict__ hi, const int16_t* __restrict__ rem,
                            float* __restrict__ master, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    master[i] = rem_join(hi[i], static_cast<uint16_t>(rem[i]));
  }
}

__global__ void q8_dequant_kernel(const QTables* __restrict__ qt, int which,
                                  const uint8_t* __restrict__ codes,
                                  const float* __restrict__ absmax, float* __restrict__ out,
                                  int64_t n) {
  const float* value = qt->map[which].value;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = __fmul_rn(value[codes[i]], absmax[i / kQBlock]);
}

// One warp per 256-element block: absmax over bit patterns, then nearest code
// of x / absmax through the same bucket search the step uses.
__global__ void q8_quant_kernel(const QTables* __restrict__ qt, int which,
                                const float* __restrict__ x, uint8_t* __restrict__ codes,
                                float* __restrict__ absmax, int64_t n) {
  const QMapDev& t = qt->map[which];
  const int refine = qt->refine;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t nblk = (n + kQBlock - 1) / kQBlock;
  for (int64_t b = blockIdx.x * (int64_t)(blockDim.x / 32) + (threadIdx.x >> 5); b < nblk;
       b += warps) {
    float v[8];
    uint32_t mx = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t e = b * kQBlock + lane * 8 + i;
      v[i] = e < n ? x[e] : 0.0f;
      mx = max(mx, __float_as_uint(v[i]) & 0x7FFFFFFFu);
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    const float A = __uint_as_float(mx);
    const float scale = A < kTinyAbsmax ? kTinyScale : 1.0f;
    const float inv = __frcp_rn(__fmul_rn(A, scale));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t e = b * kQBlock + lane * 8 + i;
      if (e >= n) continue;
      uint32_t c;
      if (mx == 0u) {
        c = static_cast<uint32_t>(qt->zero_code[which]);
      } else {
        // |q| <= 1 or NaN; NaN falls in the last bucket, which yields code 0
        const float q = __fmul_rn(__fmul_rn(v[i], scale), inv);
        const uint32_t bits = __float_as_uint(q);
        const int k = bucket_of(bits & 0x7FFFFFFFu);
        const uint32_t lo = (bits >> 31) ? t.lo_neg[k] : t.lo_pos[k];
        c = lo;
        for (int r = 0; r < refine; ++r) c += (t.thr[lo + r] <= q) ? 1u : 0u;
      }
      codes[e] = static_cast<uint8_t>(c);
    }
    if (lane == 0) absmax[b] = A;
  }
}

// lr = table[clamp(completed steps, 0, n - 1)]: one thread, stream-ordered.
__global__ void lr_from_table_kernel(const float* __restrict__ table, int32_t n,
                                     const int32_t* __restrict__ step, float* __restrict__ lr) {
  int32_t s = *step;
  s = s < 0 ? 0 : (s > n - 1 ? n - 1 : s);
  *lr = table[s];
}

int grid_for(int64_t n, int per_block) {
  int64_t g = (n + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 152 * 16) g = 152 * 16;
  return static_cast<int>(g);
}


// ---------------------------------------------------------------- 4-bit export / import
// Packed 4-bit codes (even element in the low nibble), one absmax per 128.
__global__ void q4_dequant_kernel(const QTables* __restrict__ qt, int which,
                                  const uint8_t* __restrict__ codes,
                                  const float* __restrict__ absmax, float* __restrict__ out,
                                  int64_t n) {
  const float* value = qt->map[which].value;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t c = (codes[i >> 1] >> ((i & 1) * 4)) & 0xFu;
    out[i] = __fmul_rn(value[c], absmax[i / 128]);
  }
}

// One half-warp per 128-element block (8 elements per lane): absmax over bit
// patterns by a 16-lane xor maximum, then the nearest code of x / absmax.
__global__ void q4_quant_kernel(const QTables* __restrict__ qt, int which,
                                const float* __restrict__ x, uint8_t* __restrict__ codes,
                                float* __restrict__ absmax, int64_t n) {
  const QMapDev& t = qt->map[which];
  const int refine = qt->refine;
  const int lane = threadIdx.x & 31, l16 = lane & 15;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t nblk = (n + 127) / 128;
  for (int64_t w = blockIdx.x * (int64_t)(blockDim.x / 32) + (threadIdx.x >> 5); 2 * w < nblk;
       w += warps) {
    const int64_t b = 2 * w + (lane >> 4);
    float v[8];
    uint32_t mx = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t e = b * 128 + l16 * 8 + i;
      v[i] = (b < nblk && e < n) ? x[e] : 0.0f;
      mx = max(mx, __float_as_uint(v[i]) & 0x7FFFFFFFu);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if (b >= nblk) continue;
    const float A = __uint_as_float(mx);
    const float scale = A < kTinyAbsmax ? kTinyScale : 1.0f;
    const float inv = __frcp_rn(__fmul_rn(A, scale));
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (mx == 0u) {
        q[i] = static_cast<uint32_t>(qt->zero_code[which]);
      } else {
        const float y = __fmul_rn(__fmul_rn(v[i], scale), inv);
        const uint32_t bits = __float_as_uint(y);
        const int k = bucket_of(bits & 0x7FFFFFFFu);
        const uint32_t lo = (bits >> 31) ? t.lo_neg[k] : t.lo_pos[k];
        uint32_t c = lo;
        for (int r = 0; r < refine; ++r) c += (t.thr[lo + r] <= y) ? 1u : 0u;
        q[i] = c;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const int64_t e = b * 128 + l16 * 8 + i;
      if (e < n) codes[e >> 1] = static_cast<uint8_t>(q[i] | (e + 1 < n ? q[i + 1] << 4 : 0u));
    }
    if (l16 == 0) absmax[b] = A;
  }
}

}  // namespace

cudaError_t launch_nonfinite(adamw_dtype gdt, const TensorDesc* tensors, const Chunk* chunks,
                             int64_t n_chunks, float* found_inf, int grid, cudaStream_t s) {
  switch (gdt) {
    case ADAMW_F32:
      nonfinite_kernel<ADAMW_F32><<<grid, kThreads, 0, s>>>(tensors, chunks, n_chunks, found_inf);
      break;
    case ADAMW_F16:
      nonfinite_kernel<ADAMW_F16><<<grid, kThreads, 0, s>>>(tensors, chunks, n_chunks, found_inf);
      break;
    case ADAMW_BF16:
      nonfinite_kernel<ADAMW_BF16><<<grid, kThreads, 0, s>>>(tensors, chunks, n_chunks, found_inf);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_lr_from_table(const float* table, int32_t n, const int32_t* step, float* lr,
                                 cudaStream_t s) {
  lr_from_table_kernel<<<1, 1, 0, s>>>(table, n, step, lr);
  return cudaGetLastError();
}

cudaError_t launch_split(const float* master, uint16_t* hi, int16_t* rem, int64_t n,
                         cudaStream_t s) {
  split_kernel<<<grid_for(n, kThreads), kThreads, 0, s>>>(master, hi, rem, n);
  return cudaGetLastError();
}

cudaError_t launch_join(const uint16_t* hi, const int16_t* rem, float* master, int64_t n,
                        cudaStream_t s) {
  join_kernel<<<grid_for(n, kThreads), kThreads, 0, s>>>(hi, rem, master, n);
  return cudaGetLastError();
}

cudaError_t launch_q8_dequant(const QTables* qt, int which, const uint8_t* codes,
                              const float* absmax, float* out, int64_t n, cudaStream_t s) {
  q8_dequant_kernel<<<grid_for(n, kThreads), kThreads, 0, s>>>(qt, which, codes, absmax, out, n);
  return cudaGetLastError();
}

cudaError_t launch_q8_quant(const QTables* qt, int which, const float* x, uint8_t* codes,
                            float* absmax, int64_t n, cudaStream_t s) {
  const int64_t nblk = (n + kQBlock - 1) / kQBlock;
  q8_quant_kernel<<<grid_for(nblk, kThreads / 32), kThreads, 0, s>>>(qt, which, x, codes,
                                                                    absmax, n);
  return cudaGetLastError();
}

cudaError_t launch_q4_dequant(const QTables* qt, int which, const uint8_t* codes,
                              const float* absmax, float* out, int64_t n, cudaStream_t s) {
  q4_dequant_kernel<<<grid_for(n, kThreads), kThreads, 0, s>>>(qt, which, codes, absmax, out, n);
  return cudaGetLastError();
}

cudaError_t launch_q4_quant(const QTables* qt, int which, const float* x, uint8_t* codes,
                            float* absmax, int64_t n, cudaStream_t s) {
  const int64_t nwarp = ((n + 127) / 128 + 1) / 2;
  q4_quant_kernel<<<grid_for(nwarp, kThreads / 32), kThreads, 0, s>>>(qt, which, x, codes, absmax, n);
  return cudaGetLastError();
}

}  // namespace adamw
