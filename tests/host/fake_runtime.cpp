// fake_runtime.cpp -- test harness: the plan code of libadamw (capi.cpp,
// qmap.cpp) linked for the host against a fake CUDA runtime and recording
// stand-ins for the kernel launchers, so that the CPU test suite can inspect
// the tables a plan builds (tensor table, chunk table, Adam-mini blocks) and
// the launch shapes it asks for, without a GPU.
//
// "Device" memory is host memory: cudaMalloc is aligned_alloc, cudaMemcpy is
// memcpy.  Every launcher records its arguments in a short history and does
// nothing else; the probe_* functions hand them to the test through ctypes.
#include <cuda_runtime_api.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <utility>
#include <vector>

#include "internal.h"

namespace {
int g_device = 0;
int g_sms = 152;

// Allocations made through the fake cudaMalloc: only these are real memory.
// The caller's tensors and scalars are fake addresses that nothing may touch.
std::vector<std::pair<uintptr_t, size_t>> g_allocs;

bool owned(const void* p, size_t n) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  for (const auto& r : g_allocs)
    if (a >= r.first && a + n <= r.first + r.second) return true;
  return false;
}

struct Launch {
  char kind[32];
  int mode, gdt, grid, algo;
  adamw::StepArgs a;
  adamw::MiniArgs ma;
  int64_t n;                    // element count of the helper launches
};
constexpr int kHist = 8;
Launch g_hist[kHist];          // the last launches, most recent at g_count - 1
int g_count = 0;

cudaError_t record(const char* kind, int mode, int gdt, int grid, int algo,
                   const adamw::StepArgs* a, const adamw::MiniArgs* ma, int64_t n) {
  Launch& l = g_hist[g_count % kHist];
  std::memset(&l, 0, sizeof l);
  std::strncpy(l.kind, kind, sizeof l.kind - 1);
  l.mode = mode;
  l.gdt = gdt;
  l.grid = grid;
  l.algo = algo;
  if (a) l.a = *a;
  if (ma) l.ma = *ma;
  l.n = n;
  ++g_count;
  return cudaSuccess;
}

adamw::SmallArgs g_small{};     // kernel parameters of the last small-plan launch
int g_small_smem = 0;

// back = 0: the last launch, 1: the one before, ...
const Launch& at(int back) { return g_hist[(g_count - 1 - back + 64 * kHist) % kHist]; }
}  // namespace

// ---------------------------------------------------------------- fake runtime
extern "C" {
cudaError_t cudaGetDevice(int* d) { *d = g_device; return cudaSuccess; }
cudaError_t cudaSetDevice(int d) { g_device = d; return cudaSuccess; }
cudaError_t cudaDeviceGetAttribute(int* v, cudaDeviceAttr attr, int) {
  *v = attr == cudaDevAttrMultiProcessorCount ? g_sms : 0;
  return cudaSuccess;
}
cudaError_t cudaMalloc(void** p, size_t n) {
  const size_t bytes = (n + 255) / 256 * 256 + 256;
  *p = std::aligned_alloc(256, bytes);
  if (!*p) return cudaErrorMemoryAllocation;
  g_allocs.emplace_back(reinterpret_cast<uintptr_t>(*p), bytes);
  return cudaSuccess;
}
cudaError_t cudaFree(void* p) {
  for (size_t i = 0; i < g_allocs.size(); ++i)
    if (g_allocs[i].first == reinterpret_cast<uintptr_t>(p)) {
      g_allocs.erase(g_allocs.begin() + static_cast<std::ptrdiff_t>(i));
      break;
    }
  std::free(p);
  return cudaSuccess;
}
cudaError_t cudaMemcpy(void* dst, const void* src, size_t n, cudaMemcpyKind kind) {
  // host <-> fake device: only the plan's own allocations are real memory
  if (kind == cudaMemcpyHostToDevice && !owned(dst, n)) return cudaSuccess;
  if (kind == cudaMemcpyDeviceToHost && !owned(src, n)) { std::memset(dst, 0, n); return cudaSuccess; }
  std::memcpy(dst, src, n);
  return cudaSuccess;
}
cudaError_t cudaMemset(void* p, int v, size_t n) {
  if (owned(p, n)) std::memset(p, v, n);
  return cudaSuccess;
}
cudaError_t cudaMemsetAsync(void* p, int v, size_t n, cudaStream_t) {
  if (owned(p, n)) std::memset(p, v, n);
  return cudaSuccess;
}
cudaError_t cudaDeviceSynchronize(void) { return cudaSuccess; }
cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }
const char* cudaGetErrorString(cudaError_t) { return "fake runtime error"; }
const char* cudaGetErrorName(cudaError_t) { return "cudaErrorFake"; }

// ---------------------------------------------------------------- probes
void probe_set_sms(int sms) { g_sms = sms; }
int probe_count(void) { return g_count; }
const char* probe_kind(int back) { return at(back).kind; }
int probe_grid(int back) { return at(back).grid; }
int probe_algo(int back) { return at(back).algo; }
int probe_mode(int back) { return at(back).mode; }
int64_t probe_n(int back) { return at(back).n; }
const void* probe_tensors(int back) { return at(back).a.tensors; }
const void* probe_chunks(int back) { return at(back).a.chunks; }
int64_t probe_n_chunks(int back) { return at(back).a.n_chunks; }
const void* probe_chunk_blk(int back) { return at(back).a.chunk_blk; }
const void* probe_blocks(int back) { return at(back).ma.blocks; }
const void* probe_red_chunks(int back) { return at(back).ma.red_chunks; }
int64_t probe_n_red(int back) { return at(back).ma.n_red; }
int probe_refine(int back) { return at(back).a.refine; }
const void* probe_small_args(void) { return &g_small; }
int probe_small_smem(void) { return g_small_smem; }
}

// ---------------------------------------------------------------- launchers
namespace adamw {
cudaError_t launch_step(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                        cudaStream_t) {
  return record("step", mode, gdt, grid, -1, &a, nullptr, 0);
}
cudaError_t step_occupancy(adamw_mode mode, adamw_dtype, int* bps, int* smem) {
  *bps = mode == ADAMW_MODE_Q8 ? 1 : 2;     // one 1024-thread CTA per SM in the 8-bit mode
  *smem = 0;
  return cudaSuccess;
}
cudaError_t launch_step_bulk(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                             cudaStream_t, int algo) {
  return record("bulk", mode, gdt, grid, algo, &a, nullptr, 0);
}
cudaError_t prepare_step_bulk(adamw_mode, adamw_dtype, int) { return cudaSuccess; }
cudaError_t launch_mini_reduce(adamw_dtype gdt, const StepArgs& a, const MiniArgs& ma, int grid,
                               cudaStream_t) {
  // the update launch follows: keep the reduction's record under its own kind
  record("mini_reduce", -1, gdt, grid, -1, &a, &ma, 0);
  return cudaSuccess;
}
cudaError_t launch_step_q4(adamw_dtype gdt, const StepArgs& a, int grid, cudaStream_t) {
  return record("q4", ADAMW_MODE_Q4, gdt, grid, -1, &a, nullptr, 0);
}
cudaError_t q4_occupancy(adamw_dtype, int* bps, int* smem) {
  *bps = 4;
  *smem = 0;
  return cudaSuccess;
}
cudaError_t bulk_occupancy_sqrt_div(adamw_mode, adamw_dtype, int* blocks) {
  *blocks = 2;
  return cudaSuccess;
}
cudaError_t run_wait_selftest(int, cudaStream_t, uint32_t* fault_bits, double* waited_ms) {
  if (fault_bits) *fault_bits = 0;
  if (waited_ms) *waited_ms = 0.0;
  return cudaSuccess;
}
cudaError_t launch_nonfinite(adamw_dtype gdt, const TensorDesc* tensors, const Chunk* chunks,
                             int64_t n_chunks, float*, int grid, cudaStream_t) {
  StepArgs a{};
  a.tensors = tensors;
  a.chunks = chunks;
  a.n_chunks = n_chunks;
  return record("nonfinite", -1, gdt, grid, -1, &a, nullptr, 0);
}
cudaError_t launch_split(const float*, uint16_t*, int16_t*, int64_t n, cudaStream_t) {
  return record("split", -1, -1, 0, -1, nullptr, nullptr, n);
}
cudaError_t fused_occupancy(adamw_mode, adamw_dtype, int* bps) {
  *bps = 2;
  return cudaSuccess;
}
cudaError_t launch_step_fused_amp(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                                  float*, cudaStream_t) {
  return record("fused_amp", mode, gdt, grid, -1, &a, nullptr, 0);
}
cudaError_t prepare_step_small(adamw_mode, adamw_dtype, int, int) { return cudaSuccess; }
cudaError_t launch_step_small(adamw_mode mode, adamw_dtype gdt, const SmallArgs& a, int grid,
                              int smem, bool fused, float*, cudaStream_t) {
  g_small = a;
  g_small_smem = smem;
  return record(fused ? "small_fused" : "small", mode, gdt, grid, -1, nullptr, nullptr, 0);
}
cudaError_t launch_lr_from_table(const float*, int32_t n, const int32_t*, float*, cudaStream_t) {
  return record("lr_table", -1, -1, 1, -1, nullptr, nullptr, n);
}
cudaError_t launch_join(const uint16_t*, const int16_t*, float*, int64_t n, cudaStream_t) {
  return record("join", -1, -1, 0, -1, nullptr, nullptr, n);
}
cudaError_t launch_q8_dequant(const QTables*, int, const uint8_t*, const float*, float*, int64_t n,
                              cudaStream_t) {
  return record("q8_dequant", -1, -1, 0, -1, nullptr, nullptr, n);
}
cudaError_t launch_q8_quant(const QTables*, int, const float*, uint8_t*, float*, int64_t n,
                            cudaStream_t) {
  return record("q8_quant", -1, -1, 0, -1, nullptr, nullptr, n);
}
cudaError_t launch_q4_dequant(const QTables*, int, const uint8_t*, const float*, float*, int64_t n,
                              cudaStream_t) {
  return record("q4_dequant", -1, -1, 0, -1, nullptr, nullptr, n);
}
cudaError_t launch_q4_quant(const QTables*, int, const float*, uint8_t*, float*, int64_t n,
                            cudaStream_t) {
  return record("q4_quant", -1, -1, 0, -1, nullptr, nullptr, n);
}
}  // namespace adamw
