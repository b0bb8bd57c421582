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
//
// A bounded wait of the kernel that gives up sets a bit in the array's fault
// word; calls never clear it, adamw_step_noalloc_status reads and clears it.
#include <cmath>
#include <cstdio>
#include <mutex>

#include "entry_checks.h"

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

// Validation that touches no device: arguments, and the chunk count's lower
// bound (every chunk holds at most kChunkMax elements), so that a list the
// array cannot hold is refused before anything is enqueued.
static adamw_status check_noalloc_args(const adamw_tensor* tensors, int32_t n_tensors,
                                       adamw_mode mode, adamw_dtype grad_dtype,
                                       const float* lr_dev, const int32_t* step_dev, float beta1,
                                       float beta2, float eps, const float* grad_scale_dev,
                                       const float* found_inf_dev, int64_t* total_out) {
  if (n_tensors < 0 || (n_tensors > 0 && !tensors)) return fail(ADAMW_EINVAL, "bad tensor list");
  if (n_tensors > kNoAllocMaxTensors)
    return fail(ADAMW_EINVAL, "more tensors than the static scratch holds (limit 1024)");
  adamw_status st = check_mode_dtype(mode, grad_dtype);
  if (st != ADAMW_OK) return st;
  if (mode != ADAMW_MODE_FP32 && mode != ADAMW_MODE_BF16_REM)
    return fail(ADAMW_EUNSUPPORTED, "only the fp32 and bf16+remainder modes have a no-allocation form");
  if ((st = check_step_scalars(lr_dev, step_dev, grad_scale_dev, found_inf_dev, beta1, beta2)) !=
          ADAMW_OK ||
      (st = check_eps(eps)) != ADAMW_OK)
    return st;

  const size_t psz = mode == ADAMW_MODE_BF16_REM ? 2 : 4;
  const size_t gsz = grad_dtype == ADAMW_F32 ? 4 : 2;
  int64_t total = 0, min_chunks = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const adamw_tensor& t = tensors[i];
    if (t.numel < 0) return fail(ADAMW_EINVAL, "a tensor has numel < 0");
    if (!std::isfinite(t.weight_decay))
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
    min_chunks += (t.numel + kChunkMax - 1) / kChunkMax;
    if (min_chunks > kNoAllocMaxChunks)
      return fail(ADAMW_EINVAL, "the tensor list needs more chunks than the static scratch "
                                "holds (limit 65536 chunks, about 1.07e9 elements)");
  }
  *total_out = total;
  return ADAMW_OK;
}

// The device address of the array on the current device, looked up (and the
// SM count read) on the first call made with that device current.
static adamw_status device_state(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ADAMW_EUNSUPPORTED, "device index out of range");
  DeviceState& ds = g_dev[dev];
  if (!ds.ready) {
    // The host-side symbol is only a stand-in, never an address.
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ds.scratch), g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress");
    e = cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
    ds.ready = true;
  }
  *out = &ds;
  return ADAMW_OK;
}

extern "C" adamw_status adamw_step_noalloc(const adamw_tensor* tensors, int32_t n_tensors,
                                           adamw_mode mode, adamw_dtype grad_dtype,
                                           const float* lr_dev, int32_t* step_dev, float beta1,
                                           float beta2, float eps, const float* grad_scale_dev,
                                           const float* found_inf_dev, void* stream) {
  int64_t total = 0;
  adamw_status st = check_noalloc_args(tensors, n_tensors, mode, grad_dtype, lr_dev, step_dev,
                                       beta1, beta2, eps, grad_scale_dev, found_inf_dev, &total);
  if (st != ADAMW_OK) return st;

  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* dsp = nullptr;
  if ((st = device_state(&dsp)) != ADAMW_OK) return st;
  DeviceState& ds = *dsp;
  // The plan path's bulk-staged kernel, one CTA per SM; its shared-memory
  // size is raised once per device, mode and grad dtype (no allocation).
  int& bps = ds.blocks_per_sm[mode][grad_dtype];
  cudaError_t e;
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

  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  TensorDesc* d_tensors = reinterpret_cast<TensorDesc*>(ds.scratch);
  Chunk* d_chunks = reinterpret_cast<Chunk*>(ds.scratch + kTensorBytes);
  StepScratch* d_step = reinterpret_cast<StepScratch*>(ds.scratch + kTicketOffset);
  // The array keeps whatever the previous call left: refresh both tables and
  // zero the step ticket, which must start at 0 (a launch that gave up may
  // have left it raised).  The bias-correction memo is keyed by step index
  // and betas, so a value left by another call is still right; the fault
  // word is kept for adamw_step_noalloc_status.
  if (n_tensors > 0 &&
      (e = cudaMemcpyAsync(d_tensors, g_host_tensors, sizeof(TensorDesc) * n_tensors,
                           cudaMemcpyHostToDevice, strm)) != cudaSuccess)
    return fail_cuda(e, "upload tensor table");
  if (n_chunks > 0 &&
      (e = cudaMemcpyAsync(d_chunks, g_host_chunks, sizeof(Chunk) * n_chunks,
                           cudaMemcpyHostToDevice, strm)) != cudaSuccess)
    return fail_cuda(e, "upload chunk table");
  if ((e = cudaMemsetAsync(&d_step->ticket, 0, sizeof(d_step->ticket), strm)) != cudaSuccess)
    return fail_cuda(e, "clear step ticket");

  const StepArgs a = base_step_args(d_tensors, d_chunks, n_chunks, d_step, lr_dev, step_dev,
                                    grad_scale_dev, found_inf_dev, beta1, beta2, eps);
  const int64_t resident = static_cast<int64_t>(bps) * ds.sms;
  const int grid = static_cast<int>(n_chunks < 1 ? 1 : (n_chunks < resident ? n_chunks : resident));
  e = launch_step_bulk(mode, grad_dtype, a, grid, strm, kAlgoAdamW);
  if (e != cudaSuccess) return fail_cuda(e, "launch adamw step");
  return ADAMW_OK;
}

extern "C" adamw_status adamw_step_noalloc_status(uint32_t* fault_bits) {
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* ds = nullptr;
  adamw_status st = device_state(&ds);
  if (st != ADAMW_OK) return st;
  StepScratch* d_step = reinterpret_cast<StepScratch*>(ds->scratch + kTicketOffset);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
  uint32_t bits = 0;
  if ((e = cudaMemcpy(&bits, &d_step->fault, sizeof(bits), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail_cuda(e, "read fault word");
  if (bits != 0 && (e = cudaMemset(&d_step->fault, 0, sizeof(bits))) != cudaSuccess)
    return fail_cuda(e, "clear fault word");
  if (fault_bits) *fault_bits = bits;
  if (bits != 0) {
    char buf[160];
    std::snprintf(buf, sizeof buf, "adamw_step_noalloc: a bounded wait in an earlier call gave "
                                   "up (fault bits 0x%x)", bits);
    set_last_error(buf);
    return ADAMW_ETIMEOUT;
  }
  return ADAMW_OK;
}
