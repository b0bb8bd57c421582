// internal.h -- device tables, launch arguments and the per-element update
// shared by the host plan code and the sm_103a kernels of libadamw.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "adamw.h"

namespace adamw {

// One CTA is 256 threads; every thread owns 8 consecutive elements per pass,
// so a warp covers exactly one 256-element Q8 block per pass.
constexpr int kThreads = 256;
constexpr int kVec = 8;
constexpr int kPass = kThreads * kVec;       // 2048 elements per CTA pass
// Passes whose loads a thread issues together, and the resident CTAs per SM
// the register budget targets, of the register-load fp32 / bf16+remainder
// path of the fused check + step (measured on GB300 for the plain step when it
// used this path: 2 x 2 -> 92% of copy bandwidth vs 88% for 1 x 3).
template <int MODE> struct Tune { static constexpr int unroll = 1, min_blocks = 3; };
template <> struct Tune<ADAMW_MODE_FP32> { static constexpr int unroll = 2, min_blocks = 2; };
constexpr int kChunkMax = 8 * kPass;         // chunks hold up to 16384 elements (chosen per plan)
// fp32 and bf16+remainder steps stage tiles through shared memory with bulk
// async copies (bulk_kernels.cu; 92% -> 98% of the copy bandwidth against
// 128-bit register loads).  The 8-bit and 4-bit steps load into registers:
// they are bound by instruction issue and load latency, and staging would
// spend shared-memory bandwidth that their code-table lookups need (a
// bulk-staged 8-bit step measured 5% slower, per-warp cp.async staging 24-38%
// slower).
// The bulk-staged step: 16 consumer warps and one producer warp per CTA.
constexpr int kBulkConsumers = 2 * kThreads;
constexpr int kBulkThreads = kBulkConsumers + 32;
// The 8-bit step runs one CTA of kQ8Threads per SM (64 registers a thread):
// its lane-private code tables (lane_tables.cuh, 141.7 KB) fit once per SM.
// The Adam-mini reduction: one chunk per warp, kRedWarps warps per CTA.
constexpr int kRedWarps = 8;
constexpr int kQ8Threads = 1024;
constexpr int kQ8Pass = kQ8Threads * kVec;   // 8192 elements per CTA pass
constexpr int kQBlock = ADAMW_Q8_BLOCK;      // 256
static_assert(kPass % kQBlock == 0, "chunks must hold whole Q8 blocks");
static_assert(32 * kVec == kQBlock, "one warp pass covers exactly one Q8 block");

// Chunk size of a plan: the whole list spread over the resident CTAs
// (sms x blocks per SM), rounded up to whole 256-element blocks and capped at
// kChunkMax.  Small plans then run as one balanced wave (one chunk per CTA);
// large ones get 16384-element chunks that CTAs stride over.
inline int64_t choose_chunk(int64_t total, int sms, int blocks_per_sm) {
  const int64_t resident = static_cast<int64_t>(sms) * (blocks_per_sm > 0 ? blocks_per_sm : 1);
  int64_t chunk = (total + resident - 1) / resident;
  chunk = (chunk + kQBlock - 1) / kQBlock * kQBlock;
  return chunk < kQBlock ? kQBlock : (chunk > kChunkMax ? kChunkMax : chunk);
}

// Nearest-code search tables of the 8-bit and 4-bit maps (see qmap.cpp).
constexpr int kBuckets = 1 + 25 * 128;       // |x| in [0, 2^-24) plus 25 binades x 128
constexpr int kMaxRefine = 4;                // thresholds compared per lookup, at most

// Update rules of the bulk-staged kernel.
constexpr int kAlgoAdamW = 0;
constexpr int kAlgoAdemamix = 1;
constexpr int kAlgoLion = 2;
constexpr int kAlgoMomentum = 3;  // coupled L2, one state
constexpr int kAlgoRmsprop = 4;
constexpr int kAlgoAdagrad = 5;
constexpr int kAlgoMini = 6;      // Adam-mini: v per element or shared per block
__host__ __device__ constexpr bool algo_two_state(int algo) {
  return algo == kAlgoAdamW || algo == kAlgoAdemamix || algo == kAlgoMini;
}
__host__ __device__ constexpr bool algo_coupled(int algo) {
  return algo == kAlgoMomentum || algo == kAlgoRmsprop || algo == kAlgoAdagrad;
}

struct TensorDesc {
  void* p;            // fp32 or bf16 param
  int16_t* rem;       // remainders (BF16_REM)
  const void* g;      // grads
  void* m;            // fp32 or uint8 codes
  void* v;            // fp32 or uint8 codes
  float* am;          // Q8 absmax of m per 256 block
  float* av;          // Q8 absmax of v per 256 block
  void* m2;           // AdEMAMix slow EMA (fp32), or null
  int64_t numel;
  float wd;
  int32_t vec_ok;     // all pointers 16-byte aligned
};

struct Chunk {
  int64_t start;      // first element, a multiple of the plan's chunk size
  int32_t tensor;     // index into the tensor table
  int32_t len;        // elements, 1..chunk size
};

struct QMapDev {                       // one code map and its search tables
  float value[256];                    // ascending map values (dequantisation)
  float thr[256 + kMaxRefine];         // thr[k]: smallest float nearer to value[k+1]; +inf padding
  uint8_t lo_pos[kBuckets];            // lowest code of any x >= 0 in the bucket of |x|
  uint8_t lo_neg[kBuckets];            // lowest code of any x <= 0 in the bucket of |x|
};

struct alignas(16) QTables {
  QMapDev map[2];                      // 0: signed (m), 1: unsigned (v)
  int32_t zero_code[2];
  int32_t refine;                      // thresholds to compare per lookup (1..kMaxRefine)
};
static_assert(sizeof(QTables) % 16 == 0, "QTables is copied to shared memory in 16-byte words");

// Plan-owned device words the step kernel keeps between launches.
struct StepScratch {
  uint32_t ticket;             // CTAs of the running launch that took a ticket; 0 between launches
  int32_t memo_t;              // step index whose bias corrections are memoised (0: none)
  uint32_t memo_b1, memo_b2;   // bit patterns of the betas they were computed for
  float memo_bc1;              // fl32(1 - b1^t)
  float memo_inv_sqrt_bc2;     // fl32(1 / sqrt(1 - b2^t))
  uint32_t fault;              // nonzero: a bounded wait in a kernel gave up (bit per site)
  uint32_t pad;
  // fused AMP step (grid barrier between the scan and the update); all three
  // only ever grow, so nothing is reset between launches
  unsigned long long amp_enter;   // CTAs that entered; / grid = launch index
  unsigned long long amp_arrive;  // CTAs that published their scan result
  unsigned long long amp_inf;     // 1 + index of the last launch that saw a non-finite grad
  unsigned long long pad2;
};
static_assert(sizeof(StepScratch) == 64, "StepScratch layout");

struct StepArgs {
  const TensorDesc* tensors;
  const Chunk* chunks;
  int64_t n_chunks;
  const float* lr;
  int32_t* step;
  const float* grad_scale;    // may be null
  const float* found_inf;     // may be null
  float beta1, beta2, eps;
  float beta3, alpha;         // AdEMAMix only
  StepScratch* scratch;       // plan-owned; ticket zero between launches
  const QTables* qt;          // Q8 only
  int refine;                 // Q8 only: thresholds per lookup (1, 2 or 4)
  const int32_t* chunk_blk = nullptr;   // Adam-mini: v block of each chunk (-1: v per element)
  const float* blk_r = nullptr;         // Adam-mini: fl(1/bc1) / h of each block, this step
};

// Plans small enough to sit in shared memory whole (small_kernels.cu): every
// CTA takes one piece of one tensor and stages all of it at once.  The tensor
// table travels in the kernel parameters (no dependent global loads before the
// first copy); tensor t's pieces are CTAs first_item .. first_item + its piece
// count - 1, each `piece` elements but the tensor's last.
constexpr int kSmallMaxTensors = 16;
constexpr int kSmallThreads = 1024;                 // 32 warps, each its own slice
constexpr int kSmallSmemMax = 216 * 1024;           // staged bytes per CTA, at most
struct SmallTensor {
  void* p;
  int16_t* rem;
  const void* g;
  float* m;
  float* v;
  int64_t numel;
  float wd;
  int32_t first_item;  // first CTA of this tensor
  int32_t piece;       // elements per CTA, a multiple of 8
  int32_t vec_ok;      // all pointers 16-byte aligned
};
struct SmallArgs {
  const float* lr;
  int32_t* step;
  const float* grad_scale;   // may be null
  const float* found_inf;    // may be null (the fused kernel decides the skip itself)
  StepScratch* scratch;
  float beta1, beta2, eps;
  int32_t n_tensors;
  SmallTensor t[kSmallMaxTensors];
};

// Adam-mini: one block of `len` contiguous elements sharing one v value
// (exp_avg_sq[v_index] of its tensor); its chunks are contiguous in the
// chunk table.
struct MiniBlock {
  int64_t v_index;
  int64_t first_chunk;
  int64_t len;
  int32_t tensor;
  int32_t n_chunks;
};

struct MiniArgs {
  const int64_t* red_chunks;  // chunks of the blocks longer than one element
  int64_t n_red;
  const MiniBlock* blocks;
  double* partial;            // per chunk: sum of g*g over the chunk
  uint32_t* arrived;          // per block: chunks summed this step (0 between launches)
  float* blk_r;               // per block: fl(1/bc1) / h, read by the update
};

// Bucket of a non-negative float bit pattern: 0 for |x| < 2^-24, then 128
// buckets per binade (exponent and the top 7 mantissa bits) up to [1, 2),
// everything larger in the last bucket.  (mag >> 16) is exponent * 128 plus
// those 7 bits, so the bucket is one subtraction and a clamp.
__host__ __device__ __forceinline__ int bucket_of(uint32_t mag) {
  const int k = static_cast<int>(mag >> 16) - (103 * 128 - 1);
  return k < 0 ? 0 : (k > kBuckets - 1 ? kBuckets - 1 : k);
}

// Normalisation of a block by its absmax A (both sides of the 8-bit path):
// x * fl(1/A); below 2^-64 both are scaled by 2^64 first (exact) so that the
// reciprocal cannot overflow.
constexpr float kTinyAbsmax = 5.42101086242752217e-20f;   // 2^-64
constexpr float kTinyScale = 1.84467440737095516e19f;     // 2^64

}  // namespace adamw

// Launchers implemented in the kernel translation units.
namespace adamw {
void set_last_error(const char* msg);  // message returned by adamw_last_error()
cudaError_t launch_step(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                        cudaStream_t s);
cudaError_t step_occupancy(adamw_mode mode, adamw_dtype gdt, int* blocks_per_sm,
                           int* smem_bytes);
cudaError_t launch_step_bulk(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                             cudaStream_t s, int algo);
cudaError_t prepare_step_bulk(adamw_mode mode, adamw_dtype gdt, int algo);
// Adam-mini block reduction and v update (mini_kernels.cu); the element
// update is the bulk kernel with kAlgoMini.
cudaError_t launch_mini_reduce(adamw_dtype gdt, const StepArgs& a, const MiniArgs& ma, int grid,
                               cudaStream_t s);
// 4-bit states (q4_kernels.cu).
cudaError_t launch_step_q4(adamw_dtype gdt, const StepArgs& a, int grid, cudaStream_t s);
cudaError_t q4_occupancy(adamw_dtype gdt, int* bps, int* smem);
// Resident CTAs per SM of the RMSprop / Adagrad bulk kernels (one footprint);
// call after prepare_step_bulk.
cudaError_t bulk_occupancy_sqrt_div(adamw_mode mode, adamw_dtype gdt, int* blocks);
cudaError_t run_wait_selftest(int limit_us, cudaStream_t s, uint32_t* fault_bits,
                              double* waited_ms);
cudaError_t launch_nonfinite(adamw_dtype gdt, const TensorDesc* tensors, const Chunk* chunks,
                             int64_t n_chunks, float* found_inf, int grid, cudaStream_t s);
cudaError_t launch_split(const float* master, uint16_t* hi, int16_t* rem, int64_t n,
                         cudaStream_t s);
cudaError_t fused_occupancy(adamw_mode mode, adamw_dtype gdt, int* blocks_per_sm);
cudaError_t launch_step_fused_amp(adamw_mode mode, adamw_dtype gdt, const StepArgs& a, int grid,
                                  float* found_inf_out, cudaStream_t s);
// Shared-memory-resident step of small plans (small_kernels.cu).  `fused`:
// the non-finite check and the step in one cooperative launch (found_inf_out
// written by CTA 0); otherwise a plain launch that honours a.found_inf.  The
// fused variant stages the results beside the originals (smem_fused_bytes;
// 0: the plan has no fused small path).
cudaError_t prepare_step_small(adamw_mode mode, adamw_dtype gdt, int smem_bytes,
                               int smem_fused_bytes);
cudaError_t launch_step_small(adamw_mode mode, adamw_dtype gdt, const SmallArgs& a, int grid,
                              int smem_bytes, bool fused, float* found_inf_out, cudaStream_t s);
cudaError_t launch_lr_from_table(const float* table, int32_t n, const int32_t* step, float* lr,
                                 cudaStream_t s);
cudaError_t launch_join(const uint16_t* hi, const int16_t* rem, float* master, int64_t n,
                        cudaStream_t s);
cudaError_t launch_q8_dequant(const QTables* qt, int which, const uint8_t* codes,
                              const float* absmax, float* out, int64_t n, cudaStream_t s);
cudaError_t launch_q8_quant(const QTables* qt, int which, const float* x, uint8_t* codes,
                            float* absmax, int64_t n, cudaStream_t s);
}  // namespace adamw
