// step_common.cuh -- device pieces shared by the step kernels: run-time
// scalars, the float64 bias corrections, the prologue and step ticket, the
// strict-fp32 element update, vector loads/stores and the remainder join/split.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"

namespace adamw {
namespace {

struct Scal {
  float b1, b2, omb1, omb2, eps, lr, step_size, inv_sqrt_bc2, inv_scale;
  float b3, omb3, alpha, rbc1;   // AdEMAMix: slow-EMA beta, 1 - b3, mix weight, fl(1/bc1)
  int scaled;
};

// b^t by float64 square-and-multiply; every product is one IEEE rounding.
// b^t by square-and-multiply.  The exponent is taken as an unsigned 32-bit
// count, so the loop ends after at most 32 rounds whatever the step counter
// holds (a counter the caller set negative, or one that wrapped past
// INT32_MAX, reads as a huge step: b^t = 0, bias corrections of 1).
__device__ double pow_binary(double b, int t) {
  double r = 1.0, x = b;
  for (uint32_t u = static_cast<uint32_t>(t); u != 0u; u >>= 1) {
    if (u & 1u) r = __dmul_rn(r, x);
    x = __dmul_rn(x, x);
  }
  return r;
}

// t + 1 with 32-bit wrap-around (no signed overflow).
__device__ __forceinline__ int next_step(int t) {
  return static_cast<int>(static_cast<uint32_t>(t) + 1u);
}

struct BiasCorr {
  float bc1, inv_sqrt_bc2;
};

// fl32(1 - b1^t) and fl32(1 / sqrt(1 - b2^t)), every step in float64.
__device__ BiasCorr bias_corrections(float beta1, float beta2, int t) {
  BiasCorr r;
  r.bc1 = __double2float_rn(__dsub_rn(1.0, pow_binary((double)beta1, t)));
  r.inv_sqrt_bc2 = __double2float_rn(
      __ddiv_rn(1.0, __dsqrt_rn(__dsub_rn(1.0, pow_binary((double)beta2, t)))));
  return r;
}

// The run-time scalars as loaded, before any arithmetic: a kernel can issue
// these loads, then other memory work, and finish the scalars afterwards.
struct RawScalars {
  float found, lr, gscale;
  int step;
  StepScratch memo;
};

__device__ __forceinline__ RawScalars load_scalars(const StepArgs& a) {
  RawScalars r;
  r.found = a.found_inf != nullptr ? *a.found_inf : 0.0f;
  r.step = *a.step;
  r.lr = *a.lr;
  r.gscale = a.grad_scale != nullptr ? *a.grad_scale : 1.0f;
  r.memo = *a.scratch;
  return r;
}

// Decide skip and compute the launch's float32 scalars from the loaded raw
// values.  The float64 bias corrections are taken from the plan's memo when
// the previous launch left them for this step index and these betas,
// otherwise computed here.
__device__ bool finish_scalars(const StepArgs& a, const RawScalars& r, Scal& s, int& t_out) {
  const float found = r.found, lr = r.lr, gscale = r.gscale;
  const int step = r.step;
  const StepScratch& memo = r.memo;
  if (found != 0.0f) return true;
  const int t = next_step(step);
  const BiasCorr bc = (memo.memo_t == t && memo.memo_b1 == __float_as_uint(a.beta1) &&
                       memo.memo_b2 == __float_as_uint(a.beta2))
                          ? BiasCorr{memo.memo_bc1, memo.memo_inv_sqrt_bc2}
                          : bias_corrections(a.beta1, a.beta2, t);
  s.b1 = a.beta1;
  s.b2 = a.beta2;
  s.omb1 = __fsub_rn(1.0f, a.beta1);
  s.omb2 = __fsub_rn(1.0f, a.beta2);
  s.eps = a.eps;
  s.lr = lr;
  s.inv_sqrt_bc2 = bc.inv_sqrt_bc2;
  s.step_size = __fdiv_rn(lr, bc.bc1);
  s.b3 = a.beta3;
  s.omb3 = __fsub_rn(1.0f, a.beta3);
  s.alpha = a.alpha;
  s.rbc1 = __fdiv_rn(1.0f, bc.bc1);
  s.scaled = a.grad_scale != nullptr;
  s.inv_scale = s.scaled ? __fdiv_rn(1.0f, gscale) : 1.0f;
  t_out = t;
  return false;
}

// Thread 0 of every CTA, before the CTA's barrier: read the run-time scalars
// (all loads issued together) and decide skip.
__device__ bool prologue(const StepArgs& a, Scal& s, int& t_out) {
  return finish_scalars(a, load_scalars(a), s, t_out);
}

// Thread 0 of every CTA that runs the step, after the barrier: take a ticket.
// Every CTA read *step (and the memo) before its ticket -- the fence orders
// it -- so the last CTA to take one can store t and the memo for step t + 1
// without any CTA of this launch seeing either.  Nothing waits on anything.
// take_ticket_with: the same with the next step's bias corrections already
// computed (a kernel that takes its ticket late computes them early, so the
// last CTA's epilogue is a few stores).
__device__ void take_ticket_with(const StepArgs& a, int t, const BiasCorr& nx) {
  __threadfence();
  const unsigned tk = atomicAdd(&a.scratch->ticket, 1u);
  if (tk == gridDim.x - 1) {
    *a.step = t;
    StepScratch* m = a.scratch;
    m->memo_bc1 = nx.bc1;
    m->memo_inv_sqrt_bc2 = nx.inv_sqrt_bc2;
    m->memo_b1 = __float_as_uint(a.beta1);
    m->memo_b2 = __float_as_uint(a.beta2);
    m->memo_t = next_step(t);
    atomicExch(&m->ticket, 0u);
  }
}

__device__ void take_ticket(const StepArgs& a, int t) {
  __threadfence();
  const unsigned tk = atomicAdd(&a.scratch->ticket, 1u);
  if (tk == gridDim.x - 1) {
    *a.step = t;
    const BiasCorr nx = bias_corrections(a.beta1, a.beta2, next_step(t));
    StepScratch* m = a.scratch;
    m->memo_bc1 = nx.bc1;
    m->memo_inv_sqrt_bc2 = nx.inv_sqrt_bc2;
    m->memo_b1 = __float_as_uint(a.beta1);
    m->memo_b2 = __float_as_uint(a.beta2);
    m->memo_t = next_step(t);
    atomicExch(&m->ticket, 0u);
  }
}

// The grid-wide vote of a fused check + step (one cooperative launch, all
// CTAs resident), in three parts so that a kernel can work between them.
// amp_enter: thread 0 of every CTA takes the launch index (it needs nothing
// but the launch itself, so it can be taken early).  amp_arrive: the same
// thread announces whether its CTA saw a non-finite grad (the flag is made
// visible before the arrival by the release reduction, which waits for no
// reply).  amp_await: it waits, bounded by 2 s, until every CTA of the
// launch has arrived.  The plan's three counters only ever grow, so nothing
// is reset between launches (a plan's fused launches all have the same
// grid).  CTA 0 writes the found-inf flag.  amp_await returns 0 (step), 1
// (skip) or 2 (the wait gave up: fault bit 8 set, the CTA must not store).
__device__ unsigned long long amp_enter(StepScratch* sc) {
  return atomicAdd(&sc->amp_enter, 1ull) / gridDim.x;
}

__device__ void amp_arrive(StepScratch* sc, unsigned long long launch, bool bad) {
  if (bad) atomicMax(&sc->amp_inf, launch + 1);
  asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(&sc->amp_arrive) : "memory");
}

__device__ unsigned long long amp_publish(StepScratch* sc, bool bad) {
  const unsigned long long launch = amp_enter(sc);
  amp_arrive(sc, launch, bad);
  return launch;
}

__device__ int amp_await(StepScratch* sc, unsigned long long launch, float* found_inf_out) {
  const unsigned long long target = (launch + 1) * gridDim.x;
  uint64_t t0;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t0));
  // poll with acquire loads: atomics on the counter would queue behind (and
  // delay) the other CTAs' publishing atomics on the same L2 line
  auto arrived = [&]() {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(&sc->amp_arrive) : "memory");
    return v;
  };
  while (arrived() < target) {
    __nanosleep(32);
    uint64_t t1;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t1));
    if (t1 - t0 > 2000000000ull) {
      atomicOr(&sc->fault, 8u);
      return 2;
    }
  }
  __threadfence();
  const bool skip = atomicAdd(&sc->amp_inf, 0ull) == launch + 1;
  if (blockIdx.x == 0) *found_inf_out = skip ? 1.0f : 0.0f;
  return skip ? 1 : 0;
}

__device__ int amp_grid_vote(StepScratch* sc, bool bad, float* found_inf_out) {
  return amp_await(sc, amp_publish(sc, bad), found_inf_out);
}

// SC: 1 when the grads carry a loss scale, 0 when they do not, -1 to ask
// s.scaled at run time.
template <int SC = -1>
__device__ __forceinline__ void update(float& p, float g, float& m, float& v, const Scal& s,
                                       float decay) {
  if (SC == 1 || (SC < 0 && s.scaled)) g = __fmul_rn(g, s.inv_scale);
  m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
  v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
  const float h = __fadd_rn(__fmul_rn(__fsqrt_rn(v), s.inv_sqrt_bc2), s.eps);
  const float u = __fdiv_rn(m, h);
  p = __fsub_rn(__fmul_rn(p, decay), __fmul_rn(s.step_size, u));
}

// The AdEMAMix element update (strict float32, order as in adamw.h).
__device__ __forceinline__ void update_ademamix(float& p, float g, float& m1, float& m2, float& v,
                                                const Scal& s, float decay) {
  if (s.scaled) g = __fmul_rn(g, s.inv_scale);
  m1 = __fadd_rn(__fmul_rn(s.b1, m1), __fmul_rn(s.omb1, g));
  m2 = __fadd_rn(__fmul_rn(s.b3, m2), __fmul_rn(s.omb3, g));
  v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
  const float h = __fadd_rn(__fmul_rn(__fsqrt_rn(v), s.inv_sqrt_bc2), s.eps);
  const float n = __fadd_rn(__fmul_rn(m1, s.rbc1), __fmul_rn(s.alpha, m2));
  const float u = __fdiv_rn(n, h);
  p = __fsub_rn(__fmul_rn(p, decay), __fmul_rn(s.lr, u));
}

// The Lion element update: decay first, then a step of exactly lr against the
// sign of b1*m + (1-b1)*g (0 for a zero or NaN interpolation); the state keeps
// the b2 EMA.
__device__ __forceinline__ void update_lion(float& p, float g, float& m, const Scal& s,
                                            float decay) {
  if (s.scaled) g = __fmul_rn(g, s.inv_scale);
  const float c = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
  const float sg = c > 0.0f ? 1.0f : (c < 0.0f ? -1.0f : 0.0f);
  p = __fsub_rn(__fmul_rn(p, decay), __fmul_rn(s.lr, sg));
  m = __fadd_rn(__fmul_rn(s.b2, m), __fmul_rn(s.omb2, g));
}

// Momentum, RMSprop and Adagrad: the decay joins the (unscaled) grad as
// g + p*wd when wd > 0 (coupled L2); one state st, no bias correction.
template <int ALGO>
__device__ __forceinline__ void update_coupled(float& p, float g, float& st, const Scal& s,
                                               float wd) {
  if (s.scaled) g = __fmul_rn(g, s.inv_scale);
  if (wd > 0.0f) g = __fadd_rn(g, __fmul_rn(p, wd));
  float d;
  if (ALGO == kAlgoMomentum) {
    st = __fadd_rn(__fmul_rn(s.b1, st), g);
    d = st;
  } else {
    st = ALGO == kAlgoRmsprop ? __fadd_rn(__fmul_rn(s.b1, st), __fmul_rn(s.omb1, __fmul_rn(g, g)))
                              : __fadd_rn(st, __fmul_rn(g, g));
    d = __fdiv_rn(g, __fadd_rn(__fsqrt_rn(st), s.eps));
  }
  p = __fsub_rn(p, __fmul_rn(s.lr, d));
}

// Adam-mini, an element of a block with shared v: r = fl(1/bc1) / h of the
// block; the parameter moves by lr * (m' * r) after the decay.
__device__ __forceinline__ void update_mini(float& p, float g, float& m, float r, const Scal& s,
                                            float decay) {
  if (s.scaled) g = __fmul_rn(g, s.inv_scale);
  m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
  p = __fsub_rn(__fmul_rn(p, decay), __fmul_rn(s.lr, __fmul_rn(m, r)));
}

// ---------------------------------------------------------------- loads/stores
__device__ __forceinline__ void ld8f(const float* q, float (&x)[8]) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(q));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(q) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void st8f(float* q, const float (&x)[8]) {
  __stcs(reinterpret_cast<float4*>(q), make_float4(x[0], x[1], x[2], x[3]));
  __stcs(reinterpret_cast<float4*>(q) + 1, make_float4(x[4], x[5], x[6], x[7]));
}
__device__ __forceinline__ void ld8u16(const void* q, uint32_t (&w)[4]) {
  const uint4 a = __ldcs(reinterpret_cast<const uint4*>(q));
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
}
__device__ __forceinline__ void st8u16(void* q, const uint32_t (&w)[4]) {
  __stcs(reinterpret_cast<uint4*>(q), make_uint4(w[0], w[1], w[2], w[3]));
}

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }
__device__ __forceinline__ float f16_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

template <typename GT> struct Grad;
template <> struct Grad<float> {
  static __device__ __forceinline__ void load8(const void* g, int64_t e, float (&x)[8]) {
    ld8f(static_cast<const float*>(g) + e, x);
  }
  static __device__ __forceinline__ float load1(const void* g, int64_t e) {
    return static_cast<const float*>(g)[e];
  }
};
template <> struct Grad<__half> {
  static __device__ __forceinline__ void load8(const void* g, int64_t e, float (&x)[8]) {
    uint32_t w[4];
    ld8u16(static_cast<const uint16_t*>(g) + e, w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = f16_to_f32(w[i] & 0xFFFFu);
      x[2 * i + 1] = f16_to_f32(w[i] >> 16);
    }
  }
  static __device__ __forceinline__ float load1(const void* g, int64_t e) {
    return f16_to_f32(static_cast<const uint16_t*>(g)[e]);
  }
};
template <> struct Grad<__nv_bfloat16> {
  static __device__ __forceinline__ void load8(const void* g, int64_t e, float (&x)[8]) {
    uint32_t w[4];
    ld8u16(static_cast<const uint16_t*>(g) + e, w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_to_f32(w[i] & 0xFFFFu);
      x[2 * i + 1] = bf16_to_f32(w[i] >> 16);
    }
  }
  static __device__ __forceinline__ float load1(const void* g, int64_t e) {
    return bf16_to_f32(static_cast<const uint16_t*>(g)[e]);
  }
};

// One raw grad of a shared-memory stage, widened exactly to float32.
template <typename GT>
__device__ __forceinline__ float grad_from_smem(const unsigned char* base, int idx) {
  if constexpr (sizeof(GT) == 4) {
    return reinterpret_cast<const float*>(base)[idx];
  } else {
    const uint32_t h = reinterpret_cast<const uint16_t*>(base)[idx];
    if constexpr (std::is_same<GT, __half>::value) return f16_to_f32(h);
    return bf16_to_f32(h);
  }
}

// Remainder join / split on one element (integer only; see adamw.h).
__device__ __forceinline__ float rem_join(uint32_t hi, uint32_t rem16) {
  const uint32_t top = (hi - (rem16 >> 15)) & 0xFFFFu;
  return __uint_as_float((top << 16) | (rem16 & 0xFFFFu));
}
__device__ __forceinline__ void rem_split(float x, uint32_t& hi, uint32_t& rem16) {
  uint32_t b = __float_as_uint(x);
  // a NaN master is stored as the quiet NaN 0x7FC00000: bf16 half 0x7FC0 (a
  // NaN), remainder 0 -- the increment would carry the all-ones NaNs (the
  // GPU's own 0x7FFFFFFF among them) out of the half, to -0.0 / +0.0
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) b = 0x7FC00000u;
  const uint32_t lo = b & 0xFFFFu;
  hi = ((b >> 16) + (lo >> 15)) & 0xFFFFu;
  rem16 = lo;
}

// Elements [e, e + n) one at a time: ragged tails and tensors whose pointers
// are not all 16-byte aligned.
template <adamw_mode MODE, typename GT, int ALGO = kAlgoAdamW>
__device__ void update_scalar(const TensorDesc& td, int64_t e, int n, const Scal& s,
                              float decay, float mini_r = 0.0f, bool mini_shared = false) {
  float* const pf = static_cast<float*>(td.p);
  uint16_t* const ph = static_cast<uint16_t*>(td.p);
  float* const mf = static_cast<float*>(td.m);
  float* const vf = static_cast<float*>(td.v);
  for (int i = 0; i < n; ++i) {
    const int64_t k = e + i;
    float p = MODE == ADAMW_MODE_FP32 ? pf[k] : rem_join(ph[k], static_cast<uint16_t>(td.rem[k]));
    float m = mf[k];
    const bool has_v = algo_two_state(ALGO) && !(ALGO == kAlgoMini && mini_shared);
    float v = has_v ? vf[k] : 0.0f;
    if (ALGO == kAlgoMini && mini_shared) {
      update_mini(p, Grad<GT>::load1(td.g, k), m, mini_r, s, decay);
    } else if (algo_coupled(ALGO)) {
      update_coupled<ALGO>(p, Grad<GT>::load1(td.g, k), m, s, decay);
    } else if (ALGO == kAlgoAdemamix) {
      float* const m2f = static_cast<float*>(td.m2);
      float m2 = m2f[k];
      update_ademamix(p, Grad<GT>::load1(td.g, k), m, m2, v, s, decay);
      m2f[k] = m2;
    } else if (ALGO == kAlgoLion) {
      update_lion(p, Grad<GT>::load1(td.g, k), m, s, decay);
    } else {
      update(p, Grad<GT>::load1(td.g, k), m, v, s, decay);
    }
    if (MODE == ADAMW_MODE_FP32) {
      pf[k] = p;
    } else {
      uint32_t h, r;
      rem_split(p, h, r);
      ph[k] = static_cast<uint16_t>(h);
      td.rem[k] = static_cast<int16_t>(static_cast<uint16_t>(r));
    }
    mf[k] = m;
    if (has_v) vf[k] = v;
  }
}

// ---------------------------------------------------------------- 8-bit states
// Nearest code of a normalised x (|x| <= 1, or NaN) in one map: the bucket of
// |x| gives the lowest code any x of that bucket can have; at most R
// thresholds lie inside a bucket, and code = lo + #{r < R : thr[lo + r] <= x}
// because thr is ascending.  NaN lands in the last bucket, whose lowest code
// is 0 and whose thresholds never compare true: code 0.
template <int R, bool kSigned = true>
__device__ __forceinline__ uint32_t nearest_code(float x, const QMapDev& t) {
  const uint32_t b = __float_as_uint(x);
  const int k = bucket_of(b & 0x7FFFFFFFu);
  // the second moment is never negative (a NaN of either sign reaches the last
  // bucket of either table, whose lowest code is 0): its lookups skip the sign
  const uint32_t lo = (kSigned && (b >> 31)) ? t.lo_neg[k] : t.lo_pos[k];
  uint32_t c = lo;
#pragma unroll
  for (int r = 0; r < R; ++r) c += (t.thr[lo + r] <= x) ? 1u : 0u;
  return c;
}

// Per-warp block constants for re-quantisation: the absmax bits, the scale
// (1, or 2^64 below 2^-64) and the reciprocal fl(1/(A*scale)).
struct BlockNorm {
  uint32_t bits;
  float scale, inv;
};

__device__ __forceinline__ BlockNorm block_norm(uint32_t amax_bits) {
  const float A = __uint_as_float(amax_bits);
  BlockNorm n;
  n.bits = amax_bits;
  n.scale = A < kTinyAbsmax ? kTinyScale : 1.0f;
  n.inv = __frcp_rn(__fmul_rn(A, n.scale));
  return n;
}

// Codes of the 8 values one lane owns.  All branches are warp-uniform (the
// block constants are the same in every lane); x * 1 is exact, so the
// scaled multiply is skipped when the scale is 1.
template <int R, bool kSigned = true>
__device__ __forceinline__ void quant8(const float (&x)[8], const BlockNorm& n,
                                       const QMapDev& t, uint32_t zero_code, uint32_t (&q)[8]) {
  if (n.bits == 0u) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = zero_code;
  } else if (n.scale == 1.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = nearest_code<R, kSigned>(__fmul_rn(x[i], n.inv), t);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      q[i] = nearest_code<R, kSigned>(__fmul_rn(__fmul_rn(x[i], n.scale), n.inv), t);
  }
}

__device__ __forceinline__ uint2 pack8(const uint32_t (&q)[8]) {
  return make_uint2(q[0] | q[1] << 8 | q[2] << 16 | q[3] << 24,
                    q[4] | q[5] << 8 | q[6] << 16 | q[7] << 24);
}

}  // namespace
}  // namespace adamw
