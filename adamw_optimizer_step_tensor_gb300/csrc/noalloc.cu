// noalloc.cu -- adamw_step_noalloc: one AdamW step that allocates no memory.
//
// The plan-based path (adamw_plan_create + adamw_step) keeps its tensor table,
// chunk table and step ticket in device memory that adamw_plan_create obtains
// with cudaMalloc.  Some callers cannot do that: code running while a caching
// allocator owns all free device memory, code that must not allocate in the
// middle of a training or serving loop (an allocation can synchronise the
// device or fail late under fragmentation), and embedders whose rules forbid
// any allocation outside their own pool.  For them this file keeps the same
// tables in one fixed static device array that is part of the loaded module,
// and runs the unchanged step kernel on it.
//
// Limits: at most kNoAllocMaxTensors tensors and kNoAllocMaxChunks chunks per
// call (chunks are at most 16384 elements, so up to about 1.07e9 elements);
// the array is about 1.1 MB and every GPU that loads the library holds it
// until the process exits.  fp32 and bf16+remainder modes only.
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace adamw {
namespace {

constexpr int kNoAllocMaxTensors = 1024;
constexpr int kNoAllocMaxChunks = 65536;
constexpr size_t kTensorBytes = sizeof(TensorDesc) * kNoAllocMaxTensors;
constexpr size_t kChunkBytes = sizeof(Chunk) * kNoAllocMaxChunks;
constexpr size_t kTicketOffset = kTensorBytes + kChunkBytes;
constexpr size_t kScratchBytes = kTicketOffset + 256;
static_assert(kTensorBytes % 256 == 0 && kChunkBytes % 256 == 0, "keep the parts 256-byte aligned");
constexpr int kMaxDevices = 64;

// The scratch: tensor table, chunk table, step scratch (ticket and memo).  Host code must
// never use this symbol as an address; it goes through cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceState {
  bool ready = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
  int sms = 0;
  int blocks_per_sm[3][3] = {};       // [mode][grad dtype], 0 = not queried yet
};

std::mutex g_mutex;                   // guards everything below
DeviceState g_dev[kMaxDevices];
TensorDesc g_host_tensors[kNoAllocMaxTensors];   // host staging, static: no heap use
Chunk g_host_chunks[kNoAllocMaxChunks];
// Errors are reported through adamw_last_error(), like every other entry point.
adamw_status fail(adamw_status st, const char* msg) {
  char buf[512];
  std::snprintf(buf, sizeof buf, "adamw_step_noalloc: %s", msg);
  set_last_error(buf);
  return st;
}

adamw_status fail_cuda(cudaError_t e, const char* what) {
  char buf[512];
  std::snprintf(buf, sizeof buf, "adamw_step_noalloc: %s: %s", what, cudaGetErrorString(e));
  set_last_error(buf);
  return ADAMW_ECUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace adamw

using namespace adamw;

extern "C" adamw_status adamw_step_noalloc(const adamw_tensor* tensors, int32_t n_tensors,
                                           adamw_mode mode, adamw_dtype grad_dtype,
                                           const float* lr_dev, int32_t* step_dev, float beta1,
                                           float beta2, float eps, const float* grad_scale_dev,
                                           const float* found_inf_dev, void* stream) {
  if (n_tensors < 0 || (n_tensors > 0 && !tensors)) return fail(ADAMW_EINVAL, "bad tensor list");
  if (n_tensors > kNoAllocMaxTensors)
    return fail(ADAMW_EINVAL, "more tensors than the static scratch holds (limit 1024)");
  if (mode != ADAMW_MODE_FP32 && mode != ADAMW_MODE_BF16_REM)
    return fail(ADAMW_EUNSUPPORTED, "only the fp32 and bf16+remainder modes have a no-allocation form");
  if (grad_dtype != ADAMW_F32 && grad_dtype != ADAMW_F16 && grad_dtype != ADAMW_BF16)
    return fail(ADAMW_EDTYPE, "unknown grad dtype");
  if (!lr_dev || !step_dev) return fail(ADAMW_EINVAL, "lr_dev and step_dev must be set");
  if (!aligned(lr_dev, 4) || !aligned(step_dev, 4) || !aligned(grad_scale_dev, 4) ||
      !aligned(found_inf_dev, 4))
    return fail(ADAMW_EALIGN, "a scalar pointer is not 4-byte aligned");
  if (!(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f) || !(eps >= 0.0f))
    return fail(ADAMW_EINVAL, "betas must lie in [0, 1) and eps must be >= 0");

  const size_t psz = mode == ADAMW_MODE_BF16_REM ? 2 : 4;
  const size_t gsz = grad_dtype == ADAMW_F32 ? 4 : 2;
  int64_t total = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const adamw_tensor& t = tensors[i];
    if (t.numel < 0) return fail(ADAMW_EINVAL, "a tensor has numel < 0");
    if (!(t.weight_decay == t.weight_decay) || t.weight_decay - t.weight_decay != 0.0f)
      return fail(ADAMW_EINVAL, "a tensor's weight_decay is not finite");
    if (t.numel == 0) continue;
    if (!t.param || !t.grad || !t.exp_avg || !t.exp_avg_sq || t.absmax_m || t.absmax_v ||
        (mode == ADAMW_MODE_BF16_REM) != (t.param_rem != nullptr))
      return fail(ADAMW_EINVAL, "a tensor's pointers do not match the mode");
    if (t.exp_avg_slow)
      return fail(ADAMW_EUNSUPPORTED, "AdEMAMix slow states need a plan (adamw_ademamix_step)");
    if (!aligned(t.param, psz) || !aligned(t.grad, gsz) || !aligned(t.exp_avg, 4) ||
        !aligned(t.exp_avg_sq, 4) || (t.param_rem && !aligned(t.param_rem, 2)))
      return fail(ADAMW_EALIGN, "a pointer is not aligned to its element size");
    total += t.numel;
  }

  std::lock_guard<std::mutex> lock(g_mutex);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ADAMW_EUNSUPPORTED, "device index out of range");
  DeviceState& ds = g_dev[dev];
  if (!ds.ready) {
    // Once per device, with that device current: the device address of the
    // static array (the host-side symbol is only a stand-in, never an address).
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ds.scratch), g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress");
    e = cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
    ds.ready = true;
  }
  // The plan path's bulk-staged kernel, one CTA per SM; its shared-memory
  // size is raised once per device, mode and grad dtype (no allocation).
  int& bps = ds.blocks_per_sm[mode][grad_dtype];
  if (bps == 0) {
    e = prepare_step_bulk(mode, grad_dtype, kAlgoAdamW);
    if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(bulk step)");
    bps = 1;
  }

  // Same chunking rule as a plan: the largest chunk that gives every SM work.
  const int64_t chunk = choose_chunk(total, ds.sms, bps);
  int64_t n_chunks = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const adamw_tensor& t = tensors[i];
    TensorDesc& d = g_host_tensors[i];
    d.p = t.param;
    d.rem = t.param_rem;
    d.g = t.grad;
    d.m = t.exp_avg;
    d.v = t.exp_avg_sq;
    d.am = nullptr;
    d.av = nullptr;
    d.m2 = nullptr;
    d.numel = t.numel;
    d.wd = t.weight_decay;
    d.vec_ok = aligned(t.param, 16) && aligned(t.grad, 16) && aligned(t.exp_avg, 16) &&
               aligned(t.exp_avg_sq, 16) && (!t.param_rem || aligned(t.param_rem, 16));
    for (int64_t s = 0; s < t.numel; s += chunk) {
      if (n_chunks == kNoAllocMaxChunks)
        return fail(ADAMW_EINVAL, "the tensor list needs more chunks than the static scratch "
                                  "holds (limit 65536 chunks, about 1.07e9 elements)");
      g_host_chunks[n_chunks++] =
          Chunk{s, i, static_cast<int32_t>(t.numel - s < chunk ? t.numel - s : chunk)};
    }
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TensorDesc* d_tensors = reinterpret_cast<TensorDesc*>(ds.scratch);
  Chunk* d_chunks = reinterpret_cast<Chunk*>(ds.scratch + kTensorBytes);
  StepScratch* d_step = reinterpret_cast<StepScratch*>(ds.scratch + kTicketOffset);
  // The array keeps whatever the previous call left: refresh both tables and
  // zero the step scratch (the ticket must start at 0; a zero memo is empty).
  if (n_tensors > 0 &&
      (e = cudaMemcpyAsync(d_tensors, g_host_tensors, sizeof(TensorDesc) * n_tensors,
                           cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return fail_cuda(e, "upload tensor table");
  if (n_chunks > 0 &&
      (e = cudaMemcpyAsync(d_chunks, g_host_chunks, sizeof(Chunk) * n_chunks,
                           cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return fail_cuda(e, "upload chunk table");
  if ((e = cudaMemsetAsync(d_step, 0, sizeof(StepScratch), st)) != cudaSuccess)
    return fail_cuda(e, "clear step scratch");

  StepArgs a;
  a.tensors = d_tensors;
  a.chunks = d_chunks;
  a.n_chunks = n_chunks;
  a.lr = lr_dev;
  a.step = step_dev;
  a.grad_scale = grad_scale_dev;
  a.found_inf = found_inf_dev;
  a.beta1 = beta1;
  a.beta2 = beta2;
  a.eps = eps;
  a.beta3 = 0.0f;
  a.alpha = 0.0f;
  a.scratch = d_step;
  a.qt = nullptr;
  a.refine = 1;
  const int64_t resident = static_cast<int64_t>(bps) * ds.sms;
  const int grid = static_cast<int>(n_chunks < 1 ? 1 : (n_chunks < resident ? n_chunks : resident));
  e = launch_step_bulk(mode, grad_dtype, a, grid, st, kAlgoAdamW);
  if (e != cudaSuccess) return fail_cuda(e, "launch adamw step");
  return ADAMW_OK;
}
