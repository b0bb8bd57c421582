// capi.cpp -- the extern "C" entry points of libadamw: argument validation,
// the multi-tensor plan (chunk and tensor tables on the device), and launches.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <string>
#include <vector>

#include "entry_checks.h"

namespace adamw {
void default_maps(float smap[256], float umap[256]);
void default_maps4(float smap[16], float umap[16]);
// 4-bit export / import (aux_kernels.cu)
cudaError_t launch_q4_dequant(const QTables* qt, int which, const uint8_t* codes,
                              const float* absmax, float* out, int64_t n, cudaStream_t s);
cudaError_t launch_q4_quant(const QTables* qt, int which, const float* x, uint8_t* codes,
                            float* absmax, int64_t n, cudaStream_t s);
int build_qmap(const float* value, int n, QMapDev* out);
int zero_code_of(const float* value, int n);
}  // namespace adamw

using namespace adamw;

struct adamw_plan {
  int device = -1;
  adamw_mode mode = ADAMW_MODE_FP32;
  adamw_dtype gdt = ADAMW_F32;
  int32_t n_tensors = 0;
  int64_t total_numel = 0;
  int64_t n_chunks = 0;
  int grid = 1;
  int block_threads = kThreads;   // threads per CTA of the step kernel
  int grid_check = 1;
  TensorDesc* d_tensors = nullptr;
  Chunk* d_chunks = nullptr;
  StepScratch* d_scratch = nullptr;
  QTables* d_qt = nullptr;
  int refine = 1;              // Q8: thresholds per bucket lookup of the current maps
  bool bulk = false;           // launch the bulk-staged step kernel
  // fused check + step (adamw_step_amp): its own chunk table, sized for its own
  // co-resident grid (fp32 and bf16+remainder plans only)
  Chunk* d_chunks_fused = nullptr;
  int64_t n_chunks_fused = 0;
  int grid_fused = 0;
  bool has_slow = false;       // every tensor carries an AdEMAMix slow EMA
  bool has_v = true;           // every tensor carries exp_avg_sq (false: Lion-only plan)
  int grid_sqrt_div = 1;       // grid of the RMSprop / Adagrad kernels (2 CTAs per SM)
  // Adam-mini plans (adamw_mini_plan_create): blocks sharing one v
  bool mini = false;
  int64_t n_blocks = 0, n_red = 0;
  int grid_red = 1;
  // plans small enough to sit in shared memory whole (small_kernels.cu): the
  // tensor table as kernel parameters, one piece of one tensor per CTA
  bool small = false;
  bool small_fused = false;    // adamw_step_amp takes the fused small path too
  SmallArgs small_args{};
  int small_grid = 0;
  int small_smem = 0;
  int small_smem_fused = 0;
  MiniBlock* d_blocks = nullptr;
  int32_t* d_chunk_blk = nullptr;
  int64_t* d_red_chunks = nullptr;
  double* d_partial = nullptr;
  uint32_t* d_arrived = nullptr;
  float* d_blk_r = nullptr;
};

namespace {

thread_local std::string g_err;

adamw_status fail(adamw_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

adamw_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ADAMW_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t dtype_size(adamw_dtype d) { return d == ADAMW_F32 ? 4 : 2; }

bool valid_dtype(int d) { return d == ADAMW_F32 || d == ADAMW_F16 || d == ADAMW_BF16; }
bool valid_mode(int m) {
  return m == ADAMW_MODE_FP32 || m == ADAMW_MODE_BF16_REM || m == ADAMW_MODE_Q8 ||
         m == ADAMW_MODE_Q4;
}

// Modes whose moments are stored as codes with a per-block absmax.
bool quantized(int m) { return m == ADAMW_MODE_Q8 || m == ADAMW_MODE_Q4; }

// adamw_step_amp: the largest plan the one-launch check + step serves.
constexpr int64_t kFusedAmpMaxElems = 6LL << 20;

void free_plan(adamw_plan* p) {
  if (!p) return;
  cudaFree(p->d_tensors);
  cudaFree(p->d_chunks);
  cudaFree(p->d_chunks_fused);
  cudaFree(p->d_scratch);
  cudaFree(p->d_qt);
  cudaFree(p->d_blocks);
  cudaFree(p->d_chunk_blk);
  cudaFree(p->d_red_chunks);
  cudaFree(p->d_partial);
  cudaFree(p->d_arrived);
  cudaFree(p->d_blk_r);
  delete p;
}

adamw_status check_device(const adamw_plan* p) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != p->device)
    return fail(ADAMW_EINVAL, "plan was created on device %d but device %d is current",
                p->device, dev);
  return ADAMW_OK;
}

// Checks every step entry point shares: the plan, then the run-time scalars.
adamw_status check_step(const adamw_plan* plan, const float* lr_dev, const int32_t* step_dev,
                        const float* grad_scale_dev, const float* found_inf_dev,
                        float beta1, float beta2) {
  if (!plan) return fail(ADAMW_EINVAL, "plan is NULL");
  return check_step_scalars(lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2);
}

StepArgs step_args(const adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                   const float* grad_scale_dev, const float* found_inf_dev, float beta1,
                   float beta2, float eps) {
  return base_step_args(plan->d_tensors, plan->d_chunks, plan->n_chunks, plan->d_scratch, lr_dev,
                        step_dev, grad_scale_dev, found_inf_dev, beta1, beta2, eps);
}

// The kernel parameters of a small plan's step: its tensor table and this
// call's run-time scalars.
SmallArgs small_args(const adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                     const float* grad_scale_dev, const float* found_inf_dev, float beta1,
                     float beta2, float eps) {
  SmallArgs a = plan->small_args;
  a.lr = lr_dev;
  a.step = step_dev;
  a.grad_scale = grad_scale_dev;
  a.found_inf = found_inf_dev;
  a.scratch = plan->d_scratch;
  a.beta1 = beta1;
  a.beta2 = beta2;
  a.eps = eps;
  return a;
}

// n = 256 (8-bit maps, both must contain 0.0) or 16 (the 4-bit maps; the v
// map has no zero and an all-zero block stores code 0).
adamw_status build_qtables(const float* smap, const float* umap, int n, QTables* qt) {
  std::memset(qt, 0, sizeof(QTables));
  const int r0 = build_qmap(smap, n, &qt->map[0]);
  const int r1 = build_qmap(umap, n, &qt->map[1]);
  if (r0 < 0 || r1 < 0)
    return fail(ADAMW_EINVAL, "code maps must hold %d strictly ascending finite floats "
                              "whose neighbour sums are exact in float64", n);
  qt->zero_code[0] = zero_code_of(smap, n);
  qt->zero_code[1] = zero_code_of(umap, n);
  if (n == 16 && qt->zero_code[1] < 0) qt->zero_code[1] = 0;
  if (qt->zero_code[0] < 0 || qt->zero_code[1] < 0)
    return fail(ADAMW_EINVAL, "code maps must contain 0.0");
  const int r = r0 > r1 ? r0 : r1;
  if (r > kMaxRefine)
    return fail(ADAMW_EUNSUPPORTED,
                "code maps too dense for the bucketed search (%d thresholds share a bucket, "
                "at most %d supported)", r, kMaxRefine);
  qt->refine = r < 1 ? 1 : r;
  return ADAMW_OK;
}

}  // namespace

void adamw::set_last_error(const char* msg) { g_err = msg; }

adamw_status adamw::check_mode_dtype(int mode, int grad_dtype) {
  if (!valid_mode(mode)) return fail(ADAMW_EDTYPE, "unknown mode %d", mode);
  if (!valid_dtype(grad_dtype)) return fail(ADAMW_EDTYPE, "unknown grad dtype %d", grad_dtype);
  return ADAMW_OK;
}

// The run-time scalar pointers (lr and step required, grad scale and
// found-inf optional, all 4-byte aligned) and betas in [0, 1).
adamw_status adamw::check_step_scalars(const float* lr_dev, const int32_t* step_dev,
                                       const float* grad_scale_dev, const float* found_inf_dev,
                                       float beta1, float beta2) {
  if (!lr_dev || !step_dev) return fail(ADAMW_EINVAL, "lr_dev and step_dev must be set");
  if (!aligned(lr_dev, 4) || !aligned(step_dev, 4) || !aligned(grad_scale_dev, 4) ||
      !aligned(found_inf_dev, 4))
    return fail(ADAMW_EALIGN, "a scalar pointer is not 4-byte aligned");
  if (!(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f))
    return fail(ADAMW_EINVAL, "betas must lie in [0, 1)");
  return ADAMW_OK;
}

adamw_status adamw::check_eps(float eps) {
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(ADAMW_EINVAL, "eps must be finite and >= 0");
  return ADAMW_OK;
}

static adamw_status create_plan(const adamw_tensor* tensors, int32_t n_tensors, adamw_mode mode,
                                adamw_dtype grad_dtype, const int64_t* v_block,
                                adamw_plan** out);

extern "C" {

const char* adamw_last_error(void) { return g_err.c_str(); }

int32_t adamw_abi_version(void) { return ADAMW_ABI_VERSION; }

adamw_status adamw_plan_create(const adamw_tensor* tensors, int32_t n_tensors, adamw_mode mode,
                               adamw_dtype grad_dtype, adamw_plan** out) {
  return create_plan(tensors, n_tensors, mode, grad_dtype, nullptr, out);
}

adamw_status adamw_mini_plan_create(const adamw_tensor* tensors, const int64_t* v_block,
                                    int32_t n_tensors, adamw_mode mode, adamw_dtype grad_dtype,
                                    adamw_plan** out) {
  if (n_tensors > 0 && !v_block) return fail(ADAMW_EINVAL, "v_block is NULL");
  static const int64_t kNoBlocks = 1;   // an empty list is still an Adam-mini plan
  return create_plan(tensors, n_tensors, mode, grad_dtype, v_block ? v_block : &kNoBlocks, out);
}

}  // extern "C"

static adamw_status create_plan(const adamw_tensor* tensors, int32_t n_tensors, adamw_mode mode,
                                adamw_dtype grad_dtype, const int64_t* v_block,
                                adamw_plan** out) {
  if (!out) return fail(ADAMW_EINVAL, "out is NULL");
  *out = nullptr;
  if (n_tensors < 0) return fail(ADAMW_EINVAL, "n_tensors < 0");
  if (n_tensors > 0 && !tensors) return fail(ADAMW_EINVAL, "tensors is NULL");
  if (adamw_status st = check_mode_dtype(mode, grad_dtype); st != ADAMW_OK) return st;

  const size_t psz = mode == ADAMW_MODE_BF16_REM ? 2 : 4;
  const size_t ssz = quantized(mode) ? 1 : 4;
  const size_t gsz = dtype_size(grad_dtype);
  const size_t svec = mode == ADAMW_MODE_Q8 ? 8 : (mode == ADAMW_MODE_Q4 ? 4 : 16);

  std::vector<TensorDesc> td(static_cast<size_t>(n_tensors));
  std::vector<Chunk> chunks;
  int64_t total = 0;
  int with_slow = 0, with_v = 0, sized = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const adamw_tensor& t = tensors[i];
    if (t.numel < 0) return fail(ADAMW_EINVAL, "tensor %d: numel < 0", i);
    if (!std::isfinite(t.weight_decay))
      return fail(ADAMW_EINVAL, "tensor %d: weight_decay is not finite", i);
    TensorDesc& d = td[i];
    d.p = t.param;
    d.rem = t.param_rem;
    d.g = t.grad;
    d.m = t.exp_avg;
    d.v = t.exp_avg_sq;
    d.am = t.absmax_m;
    d.av = t.absmax_v;
    d.m2 = t.exp_avg_slow;
    d.numel = t.numel;
    d.wd = t.weight_decay;
    if (t.numel == 0) continue;
    ++sized;
    if (t.exp_avg_slow) {
      ++with_slow;
      if (!aligned(t.exp_avg_slow, 4))
        return fail(ADAMW_EALIGN, "tensor %d: exp_avg_slow is not 4-byte aligned", i);
    }
    if (!t.param || !t.grad || !t.exp_avg)
      return fail(ADAMW_EINVAL, "tensor %d: param, grad and exp_avg must be set", i);
    if (t.exp_avg_sq) ++with_v;
    if ((mode == ADAMW_MODE_BF16_REM) != (t.param_rem != nullptr))
      return fail(ADAMW_EINVAL, "tensor %d: param_rem must be set exactly in BF16_REM mode", i);
    if (quantized(mode) != (t.absmax_m != nullptr && t.absmax_v != nullptr) ||
        (!quantized(mode) && (t.absmax_m || t.absmax_v)))
      return fail(ADAMW_EINVAL, "tensor %d: absmax_m/absmax_v must be set exactly in the Q8 and Q4 modes", i);
    if (!aligned(t.param, psz) || !aligned(t.grad, gsz) || !aligned(t.exp_avg, ssz) ||
        !aligned(t.exp_avg_sq, ssz) || (t.param_rem && !aligned(t.param_rem, 2)) ||
        (t.absmax_m && !aligned(t.absmax_m, 4)) || (t.absmax_v && !aligned(t.absmax_v, 4)))
      return fail(ADAMW_EALIGN, "tensor %d: a pointer is not aligned to its element size", i);
    d.vec_ok = aligned(t.param, 16) && aligned(t.grad, 16) && aligned(t.exp_avg, svec) &&
               aligned(t.exp_avg_sq, svec) && (!t.param_rem || aligned(t.param_rem, 16)) &&
               (!t.exp_avg_slow || aligned(t.exp_avg_slow, 16));
    total += t.numel;
  }
  if (with_slow != 0 && with_slow != sized)
    return fail(ADAMW_EINVAL, "exp_avg_slow must be set on every tensor or on none");
  if (with_slow && quantized(mode))
    return fail(ADAMW_EUNSUPPORTED, "AdEMAMix slow states are supported in the fp32 and "
                                    "bf16+remainder modes");
  if (with_v != 0 && with_v != sized)
    return fail(ADAMW_EINVAL, "exp_avg_sq must be set on every tensor or on none");
  if (sized && !with_v && quantized(mode))
    return fail(ADAMW_EINVAL, "the Q8 and Q4 modes need exp_avg_sq on every tensor");
  if (sized && !with_v && with_slow)
    return fail(ADAMW_EINVAL, "an AdEMAMix plan needs exp_avg_sq on every tensor");
  if (v_block) {
    if (mode != ADAMW_MODE_FP32 && mode != ADAMW_MODE_BF16_REM)
      return fail(ADAMW_EUNSUPPORTED, "Adam-mini plans cover the fp32 and bf16+remainder modes");
    if (with_slow) return fail(ADAMW_EINVAL, "an Adam-mini plan carries no exp_avg_slow");
    if (with_v != sized) return fail(ADAMW_EINVAL, "an Adam-mini plan needs exp_avg_sq on every tensor");
    for (int32_t i = 0; i < n_tensors; ++i) {
      const int64_t n = td[i].numel, b = v_block[i];
      if (n == 0) continue;
      if (b < 1 || n % b != 0)
        return fail(ADAMW_EINVAL, "tensor %d: v_block %lld must divide numel %lld", i,
                    (long long)b, (long long)n);
      if (b != 1 && b != n && b % kVec != 0)
        return fail(ADAMW_EINVAL, "tensor %d: v_block must be 1, numel or a multiple of %d", i, kVec);
    }
  }

  // Every argument is valid; only now touch the device.
  int device = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  int bps = 0, smem = 0, bps_sd = 1;
  const bool bulk = !quantized(mode);
  if (bulk) {
    e = cudaSuccess;
    for (int algo : {kAlgoLion, kAlgoMomentum, kAlgoRmsprop, kAlgoAdagrad})
      if (e == cudaSuccess) e = prepare_step_bulk(mode, grad_dtype, algo);
    if (e == cudaSuccess && (with_v || !sized)) e = prepare_step_bulk(mode, grad_dtype, kAlgoAdamW);
    if (e == cudaSuccess && (with_slow || !sized)) e = prepare_step_bulk(mode, grad_dtype, kAlgoAdemamix);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bulk step)");
    e = bulk_occupancy_sqrt_div(mode, grad_dtype, &bps_sd);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy of the RMSprop/Adagrad step");
    bps = 1;
  } else if (mode == ADAMW_MODE_Q4) {
    e = q4_occupancy(grad_dtype, &bps, &smem);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy of the 4-bit step");
  } else {
    e = step_occupancy(mode, grad_dtype, &bps, &smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  }
  if (bps < 1) bps = 1;
  const int64_t chunk = choose_chunk(total, sms, bps);
  // Adam-mini: chunks of a shared-v block stay inside it; chunk_blk maps each
  // chunk to its block (-1: v per element)
  std::vector<int32_t> chunk_blk;
  std::vector<MiniBlock> blocks;
  std::vector<int64_t> red_chunks;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const int64_t b = v_block ? v_block[i] : 1;
    if (b == 1 || td[i].numel == 0) {
      for (int64_t s = 0; s < td[i].numel; s += chunk) {
        const int64_t len = td[i].numel - s < chunk ? td[i].numel - s : chunk;
        chunks.push_back(Chunk{s, i, static_cast<int32_t>(len)});
        chunk_blk.push_back(-1);
      }
      continue;
    }
    for (int64_t b0 = 0; b0 < td[i].numel; b0 += b) {
      MiniBlock mb;
      mb.v_index = b0 / b;
      mb.first_chunk = static_cast<int64_t>(chunks.size());
      mb.len = b;
      mb.tensor = i;
      mb.n_chunks = 0;
      for (int64_t s = 0; s < b; s += chunk) {
        const int64_t len = b - s < chunk ? b - s : chunk;
        red_chunks.push_back(static_cast<int64_t>(chunks.size()));
        chunks.push_back(Chunk{b0 + s, i, static_cast<int32_t>(len)});
        chunk_blk.push_back(static_cast<int32_t>(blocks.size()));
        ++mb.n_chunks;
      }
      blocks.push_back(mb);
    }
  }
  if (blocks.size() > static_cast<size_t>(INT32_MAX))
    return fail(ADAMW_EUNSUPPORTED, "more than 2^31 - 1 Adam-mini blocks");
  // the quantised kernels walk the chunk table with a 32-bit index
  if (chunks.size() > (static_cast<size_t>(1) << 30))
    return fail(ADAMW_EUNSUPPORTED, "more than 2^30 chunks");

  std::unique_ptr<adamw_plan, void (*)(adamw_plan*)> p(new adamw_plan, free_plan);
  p->mode = mode;
  p->gdt = grad_dtype;
  p->n_tensors = n_tensors;
  p->total_numel = total;
  p->n_chunks = static_cast<int64_t>(chunks.size());

  p->device = device;
  p->bulk = bulk;
  p->block_threads = bulk ? kBulkThreads : (mode == ADAMW_MODE_Q8 ? kQ8Threads : kThreads);
  p->has_slow = with_slow != 0 || (sized == 0 && !quantized(mode));
  p->has_v = with_v != 0 || sized == 0;
  const int64_t resident = static_cast<int64_t>(bps) * sms;
  p->grid = static_cast<int>(p->n_chunks < resident ? (p->n_chunks > 0 ? p->n_chunks : 1) : resident);
  const int64_t res_sd = static_cast<int64_t>(bps_sd < 1 ? 1 : bps_sd) * sms;
  p->grid_sqrt_div =
      static_cast<int>(p->n_chunks < res_sd ? (p->n_chunks > 0 ? p->n_chunks : 1) : res_sd);
  const int64_t check_res = 8LL * sms;
  p->grid_check = static_cast<int>(p->n_chunks < check_res ? (p->n_chunks > 0 ? p->n_chunks : 1) : check_res);

  const size_t tb = td.size() * sizeof(TensorDesc), cb = chunks.size() * sizeof(Chunk);
  if (tb && (e = cudaMalloc(&p->d_tensors, tb)) != cudaSuccess)
    return fail(ADAMW_ENOMEM, "cudaMalloc(tensor table): %s", cudaGetErrorString(e));
  if (cb && (e = cudaMalloc(&p->d_chunks, cb)) != cudaSuccess)
    return fail(ADAMW_ENOMEM, "cudaMalloc(chunk table): %s", cudaGetErrorString(e));
  if ((e = cudaMalloc(&p->d_scratch, sizeof(StepScratch))) != cudaSuccess)
    return fail(ADAMW_ENOMEM, "cudaMalloc(step scratch): %s", cudaGetErrorString(e));
  if (tb && (e = cudaMemcpy(p->d_tensors, td.data(), tb, cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(e, "upload tensor table");
  if (cb && (e = cudaMemcpy(p->d_chunks, chunks.data(), cb, cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(e, "upload chunk table");
  if ((e = cudaMemset(p->d_scratch, 0, sizeof(StepScratch))) != cudaSuccess)
    return cuda_fail(e, "clear step scratch");
  if (v_block) {
    p->mini = true;
    p->n_blocks = static_cast<int64_t>(blocks.size());
    p->n_red = static_cast<int64_t>(red_chunks.size());
    // one reduction chunk per warp, the CTAs left to the hardware scheduler
    // (it balances the tail better than a resident grid walking the chunks:
    // 25.8 against 26.7 ms on the Llama-3-8B Adam-mini step)
    const int64_t red_ctas = (p->n_red + kRedWarps - 1) / kRedWarps;
    const int64_t red_max = 0x7FFFFFFF;   // beyond it the kernel's warps stride
    p->grid_red = static_cast<int>(red_ctas < 1 ? 1 : (red_ctas < red_max ? red_ctas : red_max));
    if ((e = prepare_step_bulk(mode, grad_dtype, kAlgoMini)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(Adam-mini step)");
    const size_t nb = blocks.size(), nc = chunks.size(), nr = red_chunks.size();
    if (nc && (e = cudaMalloc(&p->d_chunk_blk, nc * sizeof(int32_t))) != cudaSuccess)
      return fail(ADAMW_ENOMEM, "cudaMalloc(chunk blocks): %s", cudaGetErrorString(e));
    if (nc && (e = cudaMemcpy(p->d_chunk_blk, chunk_blk.data(), nc * sizeof(int32_t),
                              cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "upload chunk blocks");
    if (nb) {
      if ((e = cudaMalloc(&p->d_blocks, nb * sizeof(MiniBlock))) != cudaSuccess ||
          (e = cudaMalloc(&p->d_red_chunks, nr * sizeof(int64_t))) != cudaSuccess ||
          (e = cudaMalloc(&p->d_partial, nc * sizeof(double))) != cudaSuccess ||
          (e = cudaMalloc(&p->d_arrived, nb * sizeof(uint32_t))) != cudaSuccess ||
          (e = cudaMalloc(&p->d_blk_r, nb * sizeof(float))) != cudaSuccess)
        return fail(ADAMW_ENOMEM, "cudaMalloc(Adam-mini tables): %s", cudaGetErrorString(e));
      if ((e = cudaMemcpy(p->d_blocks, blocks.data(), nb * sizeof(MiniBlock),
                          cudaMemcpyHostToDevice)) != cudaSuccess ||
          (e = cudaMemcpy(p->d_red_chunks, red_chunks.data(), nr * sizeof(int64_t),
                          cudaMemcpyHostToDevice)) != cudaSuccess ||
          (e = cudaMemset(p->d_arrived, 0, nb * sizeof(uint32_t))) != cudaSuccess)
        return cuda_fail(e, "upload Adam-mini tables");
    }
  }
  if (!quantized(mode)) {
    int bpf = 0;
    if ((e = fused_occupancy(mode, grad_dtype, &bpf)) != cudaSuccess)
      return cuda_fail(e, "occupancy of the fused step");
    if (bpf < 1) bpf = 1;
    const int64_t fchunk = choose_chunk(total, sms, bpf);
    std::vector<Chunk> fchunks;
    for (int32_t i = 0; i < n_tensors; ++i)
      for (int64_t s0 = 0; s0 < td[i].numel; s0 += fchunk) {
        const int64_t len = td[i].numel - s0 < fchunk ? td[i].numel - s0 : fchunk;
        fchunks.push_back(Chunk{s0, i, static_cast<int32_t>(len)});
      }
    p->n_chunks_fused = static_cast<int64_t>(fchunks.size());
    const int64_t fres = static_cast<int64_t>(bpf) * sms;
    p->grid_fused = static_cast<int>(p->n_chunks_fused < 1 ? 1
                                     : (p->n_chunks_fused < fres ? p->n_chunks_fused : fres));
    const size_t fb = fchunks.size() * sizeof(Chunk);
    if (fb && (e = cudaMalloc(&p->d_chunks_fused, fb)) != cudaSuccess)
      return fail(ADAMW_ENOMEM, "cudaMalloc(fused chunk table): %s", cudaGetErrorString(e));
    if (fb && (e = cudaMemcpy(p->d_chunks_fused, fchunks.data(), fb, cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "upload fused chunk table");
  }
  if (!quantized(mode) && !v_block && with_v && sized > 0 && sized <= kSmallMaxTensors) {
    // the small-plan path: every tensor in pieces of `piece` elements (a
    // multiple of 8, at least 256), one per CTA, at most one CTA per SM, and
    // each piece staged whole in shared memory
    const size_t per_elem = psz + (mode == ADAMW_MODE_BF16_REM ? 2 : 0) + gsz + 8;
    int64_t piece = ((total + sms - 1) / sms + 7) / 8 * 8;
    if (piece < 256) piece = 256;
    int64_t items = 0;
    for (int guard = 0; guard < 64; ++guard) {
      items = 0;
      for (int32_t i = 0; i < n_tensors; ++i) items += (td[i].numel + piece - 1) / piece;
      if (items <= sms) break;
      piece = ((piece * items + sms - 1) / sms + 7) / 8 * 8;
    }
    const int64_t slice = ((piece / 8 * 8) + kSmallThreads / 32 * 8 - 1) / (kSmallThreads / 32 * 8) * 8;
    const int64_t smem_b = slice * (kSmallThreads / 32) * static_cast<int64_t>(per_elem);
    // the fused variant also stages its results (p [+ remainder], m, v)
    const int64_t smem_f =
        slice * (kSmallThreads / 32) *
        static_cast<int64_t>(per_elem + psz + (mode == ADAMW_MODE_BF16_REM ? 2 : 0) + 8);
    bool all_vec = true;
    for (int32_t i = 0; i < n_tensors; ++i)
      if (td[i].numel > 0 && !td[i].vec_ok) all_vec = false;
    if (items <= sms && smem_b <= kSmallSmemMax && piece <= INT32_MAX) {
      SmallArgs& sa = p->small_args;
      int32_t item = 0, k = 0;
      for (int32_t i = 0; i < n_tensors; ++i) {
        if (td[i].numel == 0) continue;
        SmallTensor& st = sa.t[k++];
        st.p = td[i].p;
        st.rem = td[i].rem;
        st.g = td[i].g;
        st.m = static_cast<float*>(td[i].m);
        st.v = static_cast<float*>(td[i].v);
        st.numel = td[i].numel;
        st.wd = td[i].wd;
        st.first_item = item;
        st.piece = static_cast<int32_t>(piece);
        st.vec_ok = td[i].vec_ok;
        item += static_cast<int32_t>((td[i].numel + piece - 1) / piece);
      }
      sa.n_tensors = k;
      p->small_grid = item;
      p->small_smem = static_cast<int>(smem_b < 16 ? 16 : smem_b);
      // the fused variant keeps one saved element per thread for the ragged
      // tails, so it takes plans whose tensors are all 16-byte aligned
      p->small_fused = all_vec && smem_f <= kSmallSmemMax;
      p->small_smem_fused = p->small_fused ? static_cast<int>(smem_f < 16 ? 16 : smem_f) : 0;
      if ((e = prepare_step_small(mode, grad_dtype, p->small_smem, p->small_smem_fused)) != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(small-plan step)");
      p->small = true;
    }
  }
  if (quantized(mode)) {
    std::unique_ptr<QTables> qt(new QTables);
    float smap[256], umap[256];
    int n = 256;
    if (mode == ADAMW_MODE_Q4) {
      // fixed maps: the 4-bit step finds the nearest v code arithmetically,
      // which holds for the map k/16 (k = 1..16) only
      default_maps4(smap, umap);
      n = 16;
    } else {
      default_maps(smap, umap);
    }
    adamw_status st = build_qtables(smap, umap, n, qt.get());
    if (st != ADAMW_OK) return st;
    p->refine = qt->refine;
    if ((e = cudaMalloc(&p->d_qt, sizeof(QTables))) != cudaSuccess)
      return fail(ADAMW_ENOMEM, "cudaMalloc(code maps): %s", cudaGetErrorString(e));
    if ((e = cudaMemcpy(p->d_qt, qt.get(), sizeof(QTables), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "upload code maps");
  }
  // The clears (scratch, Adam-mini counters) are queued on the legacy stream
  // and a copy from pageable memory may return before its DMA lands: wait for
  // them, so that a step on any stream, blocking or not, sees the whole plan.
  if ((e = cudaStreamSynchronize(cudaStreamLegacy)) != cudaSuccess)
    return cuda_fail(e, "finish the plan's uploads");
  *out = p.release();
  return ADAMW_OK;
}

extern "C" {

adamw_status adamw_plan_destroy(adamw_plan* plan) {
  if (!plan) return ADAMW_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(plan->device);
  cudaDeviceSynchronize();
  free_plan(plan);
  if (prev >= 0) cudaSetDevice(prev);
  return ADAMW_OK;
}

adamw_status adamw_plan_info(const adamw_plan* plan, int64_t* total_numel, int64_t* n_chunks,
                             int32_t* grid_blocks, int32_t* block_threads) {
  if (!plan) return fail(ADAMW_EINVAL, "plan is NULL");
  if (total_numel) *total_numel = plan->total_numel;
  if (n_chunks) *n_chunks = plan->n_chunks;
  // the launch shape of adamw_step's kernel
  if (grid_blocks) *grid_blocks = plan->small ? plan->small_grid : plan->grid;
  if (block_threads) *block_threads = plan->small ? kSmallThreads : plan->block_threads;
  return ADAMW_OK;
}

adamw_status adamw_plan_status(const adamw_plan* plan, uint32_t* fault_bits) {
  if (!plan) return fail(ADAMW_EINVAL, "plan is NULL");
  adamw_status st = check_device(plan);
  if (st != ADAMW_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  uint32_t bits = 0;
  e = cudaMemcpy(&bits, &plan->d_scratch->fault, sizeof(bits), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read fault word");
  if (fault_bits) *fault_bits = bits;
  if (bits != 0)
    return fail(ADAMW_ETIMEOUT, "a bounded wait in the step pipeline gave up (fault bits 0x%x)", bits);
  return ADAMW_OK;
}

adamw_status adamw_wait_selftest(int32_t limit_us, double* waited_ms, void* stream) {
  if (limit_us < 0 || limit_us > 5000000) return fail(ADAMW_EINVAL, "limit_us must lie in [0, 5e6]");
  uint32_t bits = 0;
  double ms = 0.0;
  cudaError_t e = run_wait_selftest(limit_us, static_cast<cudaStream_t>(stream), &bits, &ms);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test");
  if (waited_ms) *waited_ms = ms;
  if (bits != 0) return fail(ADAMW_ETIMEOUT, "the self-test wait gave up after %.3f ms", ms);
  return ADAMW_OK;
}

adamw_status adamw_check_nonfinite(const adamw_plan* plan, float* found_inf_dev, void* stream) {
  if (!plan) return fail(ADAMW_EINVAL, "plan is NULL");
  if (!found_inf_dev) return fail(ADAMW_EINVAL, "found_inf_dev is NULL");
  if (!aligned(found_inf_dev, 4)) return fail(ADAMW_EALIGN, "found_inf_dev is not 4-byte aligned");
  adamw_status st = check_device(plan);
  if (st != ADAMW_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(found_inf_dev, 0, sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(found_inf)");
  if (plan->n_chunks == 0) return ADAMW_OK;
  e = launch_nonfinite(plan->gdt, plan->d_tensors, plan->d_chunks, plan->n_chunks, found_inf_dev,
                       plan->grid_check, s);
  if (e != cudaSuccess) return cuda_fail(e, "launch nonfinite check");
  return ADAMW_OK;
}

adamw_status adamw_step(adamw_plan* plan, const float* lr_dev, int32_t* step_dev, float beta1,
                        float beta2, float eps, const float* grad_scale_dev,
                        const float* found_inf_dev, void* stream) {
  adamw_status st = check_step(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2);
  if (st == ADAMW_OK) st = check_eps(eps);
  if (st != ADAMW_OK) return st;
  if (!plan->has_v) return fail(ADAMW_EINVAL, "the plan's tensors carry no exp_avg_sq");
  if (plan->mini) return fail(ADAMW_EINVAL, "an Adam-mini plan steps with adamw_mini_step");
  if ((st = check_device(plan)) != ADAMW_OK) return st;
  cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  if (plan->small) {
    const SmallArgs sa = small_args(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1,
                                    beta2, eps);
    cudaError_t e = launch_step_small(plan->mode, plan->gdt, sa, plan->small_grid, plan->small_smem,
                                      false, nullptr, st_);
    if (e != cudaSuccess) return cuda_fail(e, "launch small-plan adamw step");
    return ADAMW_OK;
  }
  StepArgs a = step_args(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2, eps);
  a.qt = plan->d_qt;
  a.refine = plan->refine;
  cudaError_t e = plan->bulk ? launch_step_bulk(plan->mode, plan->gdt, a, plan->grid, st_, kAlgoAdamW)
                  : plan->mode == ADAMW_MODE_Q4 ? launch_step_q4(plan->gdt, a, plan->grid, st_)
                                                : launch_step(plan->mode, plan->gdt, a, plan->grid, st_);
  if (e != cudaSuccess) return cuda_fail(e, "launch adamw step");
  return ADAMW_OK;
}

adamw_status adamw_lr_from_table(const float* table, int32_t n, const int32_t* step_dev,
                                 float* lr_dev, void* stream) {
  if (n < 1) return fail(ADAMW_EINVAL, "the schedule table needs at least one entry");
  if (!table || !step_dev || !lr_dev) return fail(ADAMW_EINVAL, "NULL pointer");
  if (!aligned(table, 4) || !aligned(step_dev, 4) || !aligned(lr_dev, 4))
    return fail(ADAMW_EALIGN, "pointers must be 4-byte aligned");
  cudaError_t e = launch_lr_from_table(table, n, step_dev, lr_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ADAMW_OK : cuda_fail(e, "launch lr lookup");
}

adamw_status adamw_ademamix_step(adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                                 float beta1, float beta2, float beta3, float alpha, float eps,
                                 const float* grad_scale_dev, const float* found_inf_dev,
                                 void* stream) {
  adamw_status st = check_step(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2);
  if (st == ADAMW_OK) st = check_eps(eps);
  if (st != ADAMW_OK) return st;
  if (!plan->has_slow)
    return fail(ADAMW_EINVAL, "the plan's tensors carry no exp_avg_slow (AdEMAMix slow EMA)");
  if (!(beta3 >= 0.0f && beta3 < 1.0f)) return fail(ADAMW_EINVAL, "betas must lie in [0, 1)");
  if (!std::isfinite(alpha)) return fail(ADAMW_EINVAL, "alpha must be finite");
  if ((st = check_device(plan)) != ADAMW_OK) return st;
  StepArgs a = step_args(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2, eps);
  a.beta3 = beta3;
  a.alpha = alpha;
  cudaError_t e = launch_step_bulk(plan->mode, plan->gdt, a, plan->grid,
                                   static_cast<cudaStream_t>(stream), kAlgoAdemamix);
  if (e != cudaSuccess) return cuda_fail(e, "launch AdEMAMix step");
  return ADAMW_OK;
}

adamw_status adamw_mini_step(adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                             float beta1, float beta2, float eps, const float* grad_scale_dev,
                             const float* found_inf_dev, void* stream) {
  adamw_status st = check_step(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2);
  if (st == ADAMW_OK) st = check_eps(eps);
  if (st != ADAMW_OK) return st;
  if (!plan->mini) return fail(ADAMW_EINVAL, "the plan was not made by adamw_mini_plan_create");
  if ((st = check_device(plan)) != ADAMW_OK) return st;
  StepArgs a = step_args(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2, eps);
  a.chunk_blk = plan->d_chunk_blk;
  a.blk_r = plan->d_blk_r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (plan->n_red > 0) {
    MiniArgs ma;
    ma.red_chunks = plan->d_red_chunks;
    ma.n_red = plan->n_red;
    ma.blocks = plan->d_blocks;
    ma.partial = plan->d_partial;
    ma.arrived = plan->d_arrived;
    ma.blk_r = plan->d_blk_r;
    e = launch_mini_reduce(plan->gdt, a, ma, plan->grid_red, s);
    if (e != cudaSuccess) return cuda_fail(e, "launch Adam-mini reduction");
  }
  e = launch_step_bulk(plan->mode, plan->gdt, a, plan->grid, s, kAlgoMini);
  if (e != cudaSuccess) return cuda_fail(e, "launch Adam-mini step");
  return ADAMW_OK;
}

adamw_status adamw_lion_step(adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                             float beta1, float beta2, const float* grad_scale_dev,
                             const float* found_inf_dev, void* stream) {
  adamw_status st = check_step(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2);
  if (st != ADAMW_OK) return st;
  if (quantized(plan->mode))
    return fail(ADAMW_EUNSUPPORTED, "Lion covers the fp32 and bf16+remainder modes");
  if ((st = check_device(plan)) != ADAMW_OK) return st;
  StepArgs a = step_args(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2, 0.0f);
  cudaError_t e = launch_step_bulk(plan->mode, plan->gdt, a, plan->grid,
                                   static_cast<cudaStream_t>(stream), kAlgoLion);
  if (e != cudaSuccess) return cuda_fail(e, "launch Lion step");
  return ADAMW_OK;
}

adamw_status adamw_coupled_step(adamw_plan* plan, adamw_coupled_rule rule, const float* lr_dev,
                                int32_t* step_dev, float beta, float eps,
                                const float* grad_scale_dev, const float* found_inf_dev,
                                void* stream) {
  adamw_status st = check_step(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta, 0.0f);
  if (st == ADAMW_OK) st = check_eps(eps);
  if (st != ADAMW_OK) return st;
  int algo;
  switch (rule) {
    case ADAMW_RULE_MOMENTUM: algo = kAlgoMomentum; break;
    case ADAMW_RULE_RMSPROP: algo = kAlgoRmsprop; break;
    case ADAMW_RULE_ADAGRAD: algo = kAlgoAdagrad; break;
    default: return fail(ADAMW_EINVAL, "unknown coupled rule %d", (int)rule);
  }
  if (quantized(plan->mode))
    return fail(ADAMW_EUNSUPPORTED, "the coupled rules cover the fp32 and bf16+remainder modes");
  if ((st = check_device(plan)) != ADAMW_OK) return st;
  StepArgs a = step_args(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev,
                         rule == ADAMW_RULE_ADAGRAD ? 0.0f : beta, 0.0f, eps);
  const int grid = algo == kAlgoMomentum ? plan->grid : plan->grid_sqrt_div;
  cudaError_t e = launch_step_bulk(plan->mode, plan->gdt, a, grid,
                                   static_cast<cudaStream_t>(stream), algo);
  if (e != cudaSuccess) return cuda_fail(e, "launch coupled-L2 step");
  return ADAMW_OK;
}

adamw_status adamw_step_amp(adamw_plan* plan, const float* lr_dev, int32_t* step_dev, float beta1,
                            float beta2, float eps, const float* grad_scale_dev, float* found_inf_dev,
                            void* stream) {
  adamw_status st = check_step(plan, lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2);
  if (st == ADAMW_OK) st = check_eps(eps);
  if (st != ADAMW_OK) return st;
  if (!found_inf_dev) return fail(ADAMW_EINVAL, "found_inf_dev must be set");
  if (quantized(plan->mode))
    return fail(ADAMW_EUNSUPPORTED, "the fused check + step covers the fp32 and bf16+remainder modes");
  if (!plan->has_v) return fail(ADAMW_EINVAL, "the plan's tensors carry no exp_avg_sq");
  if (plan->mini) return fail(ADAMW_EINVAL, "an Adam-mini plan steps with adamw_mini_step");
  if ((st = check_device(plan)) != ADAMW_OK) return st;
  if (plan->small_fused) {
    // the whole plan in shared memory: grads read once, check and step in one
    // cooperative launch (every CTA resident: at most one per SM)
    const SmallArgs sa = small_args(plan, lr_dev, step_dev, grad_scale_dev, nullptr, beta1, beta2,
                                    eps);
    cudaError_t e = launch_step_small(plan->mode, plan->gdt, sa, plan->small_grid,
                                      plan->small_smem_fused, true, found_inf_dev,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cooperative launch of the small-plan fused step");
    return ADAMW_OK;
  }
  // Past a few million elements the grads no longer stay in L2 between the
  // scan and the update, and the bulk-staged step outruns the cooperative one
  // (fp16 grads on GB300: fused 33.5 us vs 35.9 us at 4 Mi elements, 57.3 vs
  // 54.5 us at 8 Mi, 655 vs 572 us at 128 Mi): run the two launches instead.
  if (plan->total_numel > kFusedAmpMaxElems) {
    st = adamw_check_nonfinite(plan, found_inf_dev, stream);
    if (st != ADAMW_OK) return st;
    return adamw_step(plan, lr_dev, step_dev, beta1, beta2, eps, grad_scale_dev, found_inf_dev,
                      stream);
  }
  // every CTA of the cooperative launch is resident at once (grid sized at plan
  // creation, with its own chunk table); the skip is decided inside the launch
  StepArgs a = step_args(plan, lr_dev, step_dev, grad_scale_dev, nullptr, beta1, beta2, eps);
  a.chunks = plan->d_chunks_fused;
  a.n_chunks = plan->n_chunks_fused;
  cudaError_t e = launch_step_fused_amp(plan->mode, plan->gdt, a, plan->grid_fused, found_inf_dev,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cooperative launch of the fused step");
  return ADAMW_OK;
}

adamw_status adamw_bf16rem_split(const float* master, uint16_t* bf16, int16_t* rem, int64_t n,
                                 void* stream) {
  if (n < 0) return fail(ADAMW_EINVAL, "n < 0");
  if (n == 0) return ADAMW_OK;
  if (!master || !bf16 || !rem) return fail(ADAMW_EINVAL, "NULL pointer");
  if (!aligned(master, 4) || !aligned(bf16, 2) || !aligned(rem, 2))
    return fail(ADAMW_EALIGN, "pointer not aligned to its element size");
  cudaError_t e = launch_split(master, bf16, rem, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ADAMW_OK : cuda_fail(e, "launch split");
}

adamw_status adamw_bf16rem_join(const uint16_t* bf16, const int16_t* rem, float* master, int64_t n,
                                void* stream) {
  if (n < 0) return fail(ADAMW_EINVAL, "n < 0");
  if (n == 0) return ADAMW_OK;
  if (!master || !bf16 || !rem) return fail(ADAMW_EINVAL, "NULL pointer");
  if (!aligned(master, 4) || !aligned(bf16, 2) || !aligned(rem, 2))
    return fail(ADAMW_EALIGN, "pointer not aligned to its element size");
  cudaError_t e = launch_join(bf16, rem, master, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ADAMW_OK : cuda_fail(e, "launch join");
}

adamw_status adamw_q8_default_maps(float signed_map[256], float unsigned_map[256]) {
  if (!signed_map || !unsigned_map) return fail(ADAMW_EINVAL, "NULL map");
  default_maps(signed_map, unsigned_map);
  return ADAMW_OK;
}

adamw_status adamw_q4_default_maps(float signed_map[16], float unsigned_map[16]) {
  if (!signed_map || !unsigned_map) return fail(ADAMW_EINVAL, "NULL output");
  default_maps4(signed_map, unsigned_map);
  return ADAMW_OK;
}

adamw_status adamw_q8_set_maps(adamw_plan* plan, const float signed_map[256],
                               const float unsigned_map[256]) {
  if (!plan) return fail(ADAMW_EINVAL, "plan is NULL");
  if (plan->mode != ADAMW_MODE_Q8 || !plan->d_qt) return fail(ADAMW_EINVAL, "plan is not in Q8 mode");
  if (!signed_map || !unsigned_map) return fail(ADAMW_EINVAL, "NULL map");
  std::unique_ptr<QTables> qt(new QTables);
  adamw_status st = build_qtables(signed_map, unsigned_map, 256, qt.get());
  if (st != ADAMW_OK) return st;
  // steps already queued on any stream read the old maps: let them finish
  // first, and let the new maps land before returning
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpy(plan->d_qt, qt.get(), sizeof(QTables), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "upload code maps");
  if ((e = cudaStreamSynchronize(cudaStreamLegacy)) != cudaSuccess)
    return cuda_fail(e, "finish the map upload");
  plan->refine = qt->refine;
  return ADAMW_OK;
}

static adamw_status q8_io_check(const adamw_plan* plan, int32_t which, const void* a,
                                const void* b, const void* c, int64_t n,
                                adamw_mode mode = ADAMW_MODE_Q8) {
  if (!plan) return fail(ADAMW_EINVAL, "plan is NULL");
  if (plan->mode != mode || !plan->d_qt)
    return fail(ADAMW_EINVAL, "plan is not in %s mode", mode == ADAMW_MODE_Q8 ? "Q8" : "Q4");
  if (which != 0 && which != 1) return fail(ADAMW_EINVAL, "which must be 0 (m) or 1 (v)");
  if (n < 0) return fail(ADAMW_EINVAL, "n < 0");
  if (n > 0 && (!a || !b || !c)) return fail(ADAMW_EINVAL, "NULL pointer");
  return check_device(plan);
}

adamw_status adamw_q8_dequant(const adamw_plan* plan, int32_t which, const uint8_t* codes,
                              const float* absmax, float* out, int64_t n, void* stream) {
  adamw_status st = q8_io_check(plan, which, codes, absmax, out, n);
  if (st != ADAMW_OK || n == 0) return st;
  if (!aligned(absmax, 4) || !aligned(out, 4)) return fail(ADAMW_EALIGN, "misaligned float pointer");
  cudaError_t e = launch_q8_dequant(plan->d_qt, which, codes, absmax, out, n,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ADAMW_OK : cuda_fail(e, "launch q8 dequant");
}

adamw_status adamw_q8_quant(const adamw_plan* plan, int32_t which, const float* x, uint8_t* codes,
                            float* absmax, int64_t n, void* stream) {
  adamw_status st = q8_io_check(plan, which, x, codes, absmax, n);
  if (st != ADAMW_OK || n == 0) return st;
  if (!aligned(absmax, 4) || !aligned(x, 4)) return fail(ADAMW_EALIGN, "misaligned float pointer");
  cudaError_t e = launch_q8_quant(plan->d_qt, which, x, codes, absmax, n,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ADAMW_OK : cuda_fail(e, "launch q8 quant");
}

adamw_status adamw_q4_dequant(const adamw_plan* plan, int32_t which, const uint8_t* codes,
                              const float* absmax, float* out, int64_t n, void* stream) {
  adamw_status st = q8_io_check(plan, which, codes, absmax, out, n, ADAMW_MODE_Q4);
  if (st != ADAMW_OK || n == 0) return st;
  if (!aligned(absmax, 4) || !aligned(out, 4)) return fail(ADAMW_EALIGN, "misaligned float pointer");
  cudaError_t e = launch_q4_dequant(plan->d_qt, which, codes, absmax, out, n,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ADAMW_OK : cuda_fail(e, "launch q4 dequant");
}

adamw_status adamw_q4_quant(const adamw_plan* plan, int32_t which, const float* x, uint8_t* codes,
                            float* absmax, int64_t n, void* stream) {
  adamw_status st = q8_io_check(plan, which, x, codes, absmax, n, ADAMW_MODE_Q4);
  if (st != ADAMW_OK || n == 0) return st;
  if (!aligned(absmax, 4) || !aligned(x, 4)) return fail(ADAMW_EALIGN, "misaligned float pointer");
  cudaError_t e = launch_q4_quant(plan->d_qt, which, x, codes, absmax, n,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ADAMW_OK : cuda_fail(e, "launch q4 quant");
}

}  // extern "C"
