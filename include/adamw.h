/*
 * adamw.h -- C ABI of libadamw: a fused AdamW optimizer step for sm_103a (GB300).
 *
 * The step follows "Fix decoupled weight decay ordering in the CUDA
 * Adam/AdEMAMix kernels" (bitsandbytes PR #2040), PR description: weight decay
 * and the gradient-based update are both taken from the previous parameter,
 *     p <- p * (1 - lr*wd) - (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps),
 * with m <- b1*m + (1-b1)*g, v <- b2*v + (1-b2)*g*g, bc1 = 1 - b1^t,
 * bc2 = 1 - b2^t, and eps added after the bias correction of sqrt(v) as in the
 * AdamW branch of the AdamWMini listing on "Adam-mini <> DTensor".
 *
 * Arithmetic contract.  Every element is updated in float32 with exactly one
 * IEEE round-to-nearest-even rounding per operation, no fused multiply-add,
 * in this order:
 *     g  = g_raw [* inv_scale]        inv_scale = 1 / *grad_scale_dev
 *     m' = b1*m + (1-b1)*g
 *     v' = b2*v + (1-b2)*(g*g)
 *     u  = m' / (sqrt(v') * inv_sqrt_bc2 + eps)
 *     p' = p*(1 - lr*wd) - (lr/bc1)*u
 * where b^t is float64 square-and-multiply, and bc1 = 1 - b1^t and
 * inv_sqrt_bc2 = 1 / sqrt(1 - b2^t) are float64 values rounded once to
 * float32 (the bias correction of sqrt(v) is a multiplication by its
 * reciprocal rather than a per-element division).
 * Results are therefore reproducible bit for bit by any IEEE float32
 * implementation of the same sequence.  The other rules (AdEMAMix, Lion, the
 * coupled-L2 rules, Adam-mini) and the 8-bit and 4-bit modes state their own
 * sequences below in the same terms.  The library's two fused multiply-adds
 * change no result: the exact split of a square in the Adam-mini block
 * reduction, and 16x - 1.5 in the 4-bit v code search, where 16x is exact so
 * the fused and the unfused forms round the same value once.
 *
 * Conventions shared by all entry points
 *   - Every tensor, scalar and stream is owned by the caller.  Pointers named
 *     *_dev and all tensor pointers are device pointers on the device that
 *     was current when the plan was created.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Device work is asynchronous on it; no entry point that takes
 *     a stream allocates memory, and none synchronises the host except
 *     adamw_step_noalloc (its table upload is a pageable copy) and the
 *     self-test.
 *   - Arguments are validated before any launch; a non-OK status means
 *     nothing was enqueued.  adamw_last_error() returns a message for the
 *     last non-OK status of the calling thread.  Nothing is thrown across
 *     the ABI.
 *   - A plan must not be used by two steps that may run concurrently (it
 *     holds a small device counter used to advance the step count).
 */
#ifndef ADAMW_GB300_H
#define ADAMW_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ADAMW_ABI_VERSION 3
#define ADAMW_Q8_BLOCK 256
#define ADAMW_Q4_BLOCK 128

typedef enum {
  ADAMW_OK = 0,
  ADAMW_EINVAL = 1,       /* null/negative/inconsistent argument */
  ADAMW_EALIGN = 2,       /* a pointer is not aligned to its element size */
  ADAMW_EDTYPE = 3,       /* unknown dtype or mode value */
  ADAMW_ENOMEM = 4,       /* plan allocation failed */
  ADAMW_ECUDA = 5,        /* a CUDA runtime call or launch failed */
  ADAMW_EUNSUPPORTED = 6, /* a valid but unsupported combination */
  ADAMW_ETIMEOUT = 7      /* a bounded device-side wait gave up (see adamw_plan_status) */
} adamw_status;

typedef enum { ADAMW_F32 = 0, ADAMW_F16 = 1, ADAMW_BF16 = 2 } adamw_dtype;

/* Parameter / state storage of every tensor in a plan. */
typedef enum {
  /* fp32 param, fp32 m and v. */
  ADAMW_MODE_FP32 = 0,
  /* bf16 model param plus an int16 remainder per element that together hold
   * the fp32 master exactly ("Support store_param_remainders feature from
   * Apex in TE Fused Adam #1408", Description; a NaN master as the quiet NaN,
   * see adamw_bf16rem_split); fp32 m and v.  The pair is
   * joined to the fp32 master, updated, and split again in registers; the
   * split is adamw_bf16rem_split's. */
  ADAMW_MODE_BF16_REM = 1,
  /* fp32 param; m and v stored as uint8 codes into a signed (m) and an
   * unsigned (v) 256-entry code map with one fp32 absmax per 256-element
   * block of each tensor (the 8-bit blockwise 2-state step named in the
   * bitsandbytes PR above).  Per block: dequantise, update with the
   * unquantised m', v', then absmax = max|m'| and code = nearest map entry
   * to m' * fl(1/absmax) -- one reciprocal per block, a reading taken for
   * speed; it moves a code by one from the nearest entry to the correctly
   * rounded fl(m'/absmax) only where that ratio lies within 2.5 ulp of the
   * midpoint between two entries (exact tie -> lower code; all-zero block ->
   * absmax 0 and the code of 0.0). */
  ADAMW_MODE_Q8 = 2,
  /* The Q8 step with 4-bit codes and 128-element blocks (the 4-bit AdamW of
   * torchao named in "4 bit Adam should support non constant lr"; format of
   * Li, Chen, Zhu, "Memory Efficient Optimizers with 4-bit States"): m on a
   * 16-entry signed dynamic map, v on k/16 (k = 1..16, no zero; an all-zero
   * block stores absmax 0 and code 0).  exp_avg and exp_avg_sq are uint8
   * [ceil(numel/2)], two codes per byte, the even element in the low nibble
   * (an odd numel leaves the last high nibble 0); absmax_m/absmax_v fp32
   * [ceil(numel/128)].  The maps are fixed (adamw_q4_default_maps). */
  ADAMW_MODE_Q4 = 3
} adamw_mode;

/* One parameter tensor, flat and contiguous (numel elements). */
typedef struct {
  void* param;          /* fp32 [numel]; bf16 [numel] in BF16_REM mode       */
  int16_t* param_rem;   /* BF16_REM: int16 [numel]; otherwise must be NULL    */
  const void* grad;     /* grad_dtype [numel], possibly loss-scaled           */
  void* exp_avg;        /* m: fp32 [numel]; uint8 codes [numel] in Q8 mode;
                           packed 4-bit codes [ceil(numel/2)] in Q4 mode      */
  void* exp_avg_sq;     /* v: fp32 [numel]; uint8 codes [numel] in Q8 mode.
                           May be NULL on every tensor of an fp32 or
                           bf16+remainder plan: such a plan runs only the
                           1-state steps adamw_lion_step and
                           adamw_coupled_step (the others return EINVAL)     */
  float* absmax_m;      /* Q8: fp32 [ceil(numel/256)]; Q4: [ceil(numel/128)];
                           otherwise NULL                                      */
  float* absmax_v;      /* as absmax_m                                         */
  int64_t numel;        /* >= 0; tensors with numel 0 are ignored             */
  float weight_decay;   /* per tensor (e.g. 0 for norms and biases)           */
  void* exp_avg_slow;   /* AdEMAMix slow EMA m2: fp32 [numel] on every tensor of
                           the plan, or NULL on every tensor (AdamW only)      */
} adamw_tensor;

typedef struct adamw_plan adamw_plan;

/*
 * Build a plan for a fixed tensor list: validates every tensor, splits the
 * list into chunks of contiguous elements, and uploads the chunk and tensor
 * tables (and, in Q8 mode, the default code maps) to the current device.
 * The multi-tensor chunk list plays the role of the multi_tensor_adam lists
 * on the TransformerEngine page: one launch covers every tensor.
 * Pointers must be aligned to their element size (EALIGN otherwise); tensors
 * whose pointers are all 16-byte aligned take the 128-bit vector path, the
 * rest a scalar path.  Synchronous (allocates device memory and copies).
 * On success *out owns the device tables until adamw_plan_destroy.
 * An fp32 or bf16+remainder plan with exp_avg_sq, at most 16 non-empty
 * tensors and few enough elements that one piece per SM (every tensor cut
 * into pieces of equal length, a multiple of 8) fits in 216 KB of shared
 * memory -- about two million elements -- is a small plan: adamw_step and
 * adamw_step_amp then stage each piece whole in one CTA's shared memory, with
 * the tensor table passed as kernel parameters.  Same results either way.
 */
adamw_status adamw_plan_create(const adamw_tensor* tensors, int32_t n_tensors,
                               adamw_mode mode, adamw_dtype grad_dtype,
                               adamw_plan** out);

/* Free a plan (NULL is allowed).  Synchronises with the device first. */
adamw_status adamw_plan_destroy(adamw_plan* plan);

/* Plan facts for logging: element count, chunk count, and the launch shape
 * of the plan's step kernel (grid, threads per CTA; the fused AMP step and
 * the rules other than AdamW may launch other shapes).  Any output pointer
 * may be NULL. */
adamw_status adamw_plan_info(const adamw_plan* plan, int64_t* total_numel,
                             int64_t* n_chunks, int32_t* grid_blocks,
                             int32_t* block_threads);

/*
 * Device-side health of a plan.  The fp32 and bf16+remainder steps stage
 * tiles through shared memory with asynchronous bulk copies; every wait of
 * that pipeline is bounded (2 s), and a wait that gives up records a bit in
 * the plan's fault word and ends its CTA without touching further data.
 * Waits for all work on the device, then copies the word to *fault_bits
 * (may be NULL): ADAMW_OK if it is 0, ADAMW_ETIMEOUT otherwise.  The word
 * stays set until the plan is destroyed.
 */
adamw_status adamw_plan_status(const adamw_plan* plan, uint32_t* fault_bits);

/*
 * Self-test of the bounded wait used by the pipeline: one thread waits on an
 * mbarrier phase that nothing completes, for limit_us microseconds.  Returns
 * ADAMW_ETIMEOUT when the wait gave up as it must (the normal result) and
 * writes the time waited to *waited_ms; the CUDA context stays usable.
 * Synchronous on `stream`.
 */
adamw_status adamw_wait_selftest(int32_t limit_us, double* waited_ms, void* stream);

/*
 * found_inf: "FusedAdam & PyTorch Lightning AMP" -- a fused step does the
 * grad unscale itself and needs to know whether any grad is non-finite.
 * Writes 0.0f to *found_inf_dev, then 1.0f if any raw grad element of the
 * plan is +-inf or NaN.  Two stream-ordered operations (a 4-byte memset and
 * one launch); the caller may instead supply its own flag to adamw_step.
 */
adamw_status adamw_check_nonfinite(const adamw_plan* plan, float* found_inf_dev,
                                   void* stream);

/*
 * One AdamW step over every tensor of the plan, in one launch.
 *   lr_dev         device fp32 learning rate, read by the kernel at run time,
 *                  so a per-step schedule only rewrites 4 bytes (or points at
 *                  another entry of a device schedule table) and nothing is
 *                  rebuilt ("4 bit Adam should support non constant lr").
 *   step_dev       device int32 count of completed steps; this step uses
 *                  t = *step_dev + 1 and stores t there unless skipped.
 *   beta1, beta2   in [0, 1); eps finite and >= 0 (float32); EINVAL otherwise.
 *   grad_scale_dev NULL, or device fp32 loss scale: grads are multiplied by
 *                  1 / *grad_scale_dev before use.
 *   found_inf_dev  NULL, or device fp32 flag: when non-zero at run time the
 *                  whole step is skipped -- params, states, absmax and
 *                  *step_dev are left untouched.
 */
adamw_status adamw_step(adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                        float beta1, float beta2, float eps,
                        const float* grad_scale_dev, const float* found_inf_dev,
                        void* stream);

/*
 * adamw_step_noalloc -- one AdamW step over a tensor list without any memory
 * allocation.  The pages have no counterpart: this entry point exists for
 * callers that cannot call cudaMalloc (a caching allocator already owns the
 * free device memory, an allocation inside the training or serving loop is
 * not allowed because it can synchronise or fail late, or an embedding
 * application permits no allocation outside its own pool), and therefore
 * cannot build a plan.
 *
 * Arguments are those of adamw_plan_create followed by those of adamw_step,
 * with the same meaning, validation and arithmetic; the result of a call is
 * bit-identical to adamw_plan_create + adamw_step on the same inputs.  Modes
 * ADAMW_MODE_FP32 and ADAMW_MODE_BF16_REM only (EUNSUPPORTED for the 8-bit
 * and 4-bit modes, EDTYPE for an unknown mode or grad dtype).
 *
 * Instead of plan memory the call uses one static device array built into the
 * library (about 1.1 MB on every GPU that loads it, held until the process
 * exits).  Limits: at most 1024 tensors and 65536 chunks per call (a chunk
 * holds at most 16384 elements, so about 1.07e9 elements in all); larger lists
 * are rejected with ADAMW_EINVAL before anything is enqueued.  Each call
 * copies the tensor and chunk tables from a static host buffer into the array
 * (a pageable host-to-device copy, which may make the host wait for the
 * stream) and clears the array's step ticket, then launches the step kernel.
 * The first call on each device looks up the array's device address with that
 * device current; make that first call before any stream capture.  All calls
 * share the one array and it keeps what the last call left: calls whose work
 * may overlap on the GPU (different streams without ordering between them)
 * race and must not be issued.
 *
 * A bounded wait of the step kernel that gives up (2 s; a partly applied step)
 * sets a bit in the array's fault word, which no call clears; read it with
 * adamw_step_noalloc_status.
 */
adamw_status adamw_step_noalloc(const adamw_tensor* tensors, int32_t n_tensors,
                                adamw_mode mode, adamw_dtype grad_dtype,
                                const float* lr_dev, int32_t* step_dev,
                                float beta1, float beta2, float eps,
                                const float* grad_scale_dev, const float* found_inf_dev,
                                void* stream);

/*
 * The fault word of adamw_step_noalloc's static array on the current device
 * (the pages have no counterpart): synchronises the device, stores the bits
 * in *fault_bits (if not NULL), clears them, and returns ADAMW_ETIMEOUT when
 * any was set (a bounded wait of an earlier call gave up and that step may be
 * partly applied), else ADAMW_OK.  Allocates nothing.
 */
adamw_status adamw_step_noalloc_status(uint32_t* fault_bits);

/*
 * One AdEMAMix step over every tensor of the plan (plans whose tensors all
 * carry exp_avg_slow; fp32 and bf16+remainder modes).  "Fix decoupled weight
 * decay ordering in the CUDA Adam/AdEMAMix kernels" (bitsandbytes PR #2040):
 * like AdamW, decay and update both take the previous parameter; the update
 * rule is that of Pagliardini et al. (arXiv:2409.03137):
 *     m1' = b1*m1 + (1-b1)*g,  m2' = b3*m2 + (1-b3)*g,  v' = b2*v + (1-b2)*g*g
 *     p'  = p*(1 - lr*wd) - lr * (m1'/bc1 + alpha*m2') / (sqrt(v')/sqrt(bc2) + eps)
 * (the slow EMA m2 is not bias-corrected; alpha and beta3 are this step's
 * values, any warm-up schedule is the caller's).  Float32 sequence:
 *     g = g_raw [* inv_scale]; m1', m2', v' as above (one rounding per op);
 *     h = sqrt(v') * inv_sqrt_bc2 + eps;  n = m1' * fl(1/bc1) + alpha * m2';
 *     u = n / h;  p' = p*(1 - lr*wd) - lr*u.
 * Other arguments, skip and step-count semantics as adamw_step.
 */
adamw_status adamw_ademamix_step(adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                                 float beta1, float beta2, float beta3, float alpha, float eps,
                                 const float* grad_scale_dev, const float* found_inf_dev,
                                 void* stream);

/*
 * One Lion step over every tensor of the plan (fp32 and bf16+remainder
 * modes; exp_avg_sq and exp_avg_slow, if the plan has them, are neither read
 * nor written).  "Fix decoupled weight decay ordering in the CUDA
 * Adam/AdEMAMix kernels" (bitsandbytes PR #2040), review of the 1-state
 * kernels: Lion decays the parameter before its sign update.  The update is
 * that of Chen et al., "Symbolic Discovery of Optimization Algorithms"
 * (arXiv:2302.06675), with one state m and no bias correction:
 *     c  = b1*m + (1-b1)*g
 *     p' = p*(1 - lr*wd) - lr*sign(c)      sign(0) = sign(NaN) = 0
 *     m' = b2*m + (1-b2)*g
 * Float32 sequence, one rounding per operation: g = g_raw [* inv_scale];
 * c = b1*m + fl(1-b1)*g; p' = p*fl(1 - fl(lr*wd)) - lr*sign(c);
 * m' = b2*m + fl(1-b2)*g.  Reads p (+ rem), g, m and writes p (+ rem), m:
 * 20 bytes per element with fp32 params and grads.
 * lr_dev, step_dev, grad_scale_dev, found_inf_dev, skip and step counting as
 * adamw_step (*step_dev advances although Lion has no bias correction).
 * EINVAL for betas outside [0, 1); EUNSUPPORTED for 8-bit and 4-bit plans.
 */
adamw_status adamw_lion_step(adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                             float beta1, float beta2, const float* grad_scale_dev,
                             const float* found_inf_dev, void* stream);

/*
 * Adam-mini plan ("Adam-mini <> DTensor", the AdamWMini listing): like
 * adamw_plan_create (fp32 and bf16+remainder modes), plus one block length per
 * tensor, v_block[i]: the elements of tensor i form blocks of v_block[i]
 * contiguous elements that share one second moment, and exp_avg_sq of that
 * tensor holds numel / v_block[i] fp32 values.  1 gives the listing's AdamW
 * branch (embeddings and the output layer), a head's dim*dim/n_heads elements
 * its query/key branch, numel its one-v-per-tensor branch; the partition is
 * the caller's.  v_block[i] must divide numel and be 1, numel or a multiple
 * of 8 (EINVAL otherwise); exp_avg_sq is required on every tensor and
 * exp_avg_slow must be NULL.  Chunks never straddle blocks.  Such a plan steps
 * with adamw_mini_step (and, touching no v, adamw_lion_step and
 * adamw_coupled_step); adamw_step and adamw_step_amp return EINVAL.
 */
adamw_status adamw_mini_plan_create(const adamw_tensor* tensors, const int64_t* v_block,
                                    int32_t n_tensors, adamw_mode mode, adamw_dtype grad_dtype,
                                    adamw_plan** out);

/*
 * One Adam-mini step: two launches on `stream`.  The first sums g*g over
 * every block longer than one element (each 32 squares as an error-free pair
 * of float32 -- exact squares by fma, or exact as they are for unscaled
 * 16-bit grads, TwoSum additions, after Ogita, Rump and Oishi -- the pairs
 * added in float64 in a fixed order, the block's chunks in chunk order), then
 * per block, one rounding per operation:
 *     mean = fl32(sum / len);  v' = b2*v + fl(1-b2)*mean
 *     h = sqrt(v')*fl32(1/sqrt(1-b2^t)) + eps;  r = fl(1/fl32(1-b1^t)) / h
 * The second updates every element:
 *     block of 1: exactly adamw_step's sequence
 *     longer:     g = g_raw [* inv_scale];  m' = b1*m + fl(1-b1)*g
 *                 p' = p*decay - lr*(m'*r)
 * with decay = fl(1 - fl(lr*wd)) when wd > 0 and no decay otherwise (the
 * listing decays only for wd > 0).  The sum's relative error stays below
 * about 2^-37 (32 squares per float32 pair), so the mean is the correctly
 * rounded mean of the squares except within that distance of a float32
 * rounding boundary (one ulp off then).  A round of 32 squares whose float32
 * pair is not finite (a NaN or infinite grad, a square or a partial sum past
 * the float32 range) is summed again with float64 squares, so such blocks get
 * the float64 definition's inf, NaN or finite mean; squares below about
 * 2^-100, where the float32 split of a square stops being exact, may each
 * lose up to 2^-149.  lr_dev, step_dev, grad_scale_dev, found_inf_dev, skip
 * (both launches) and step counting (the second launch) as adamw_step.
 */
adamw_status adamw_mini_step(adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                             float beta1, float beta2, float eps, const float* grad_scale_dev,
                             const float* found_inf_dev, void* stream);

/* The 1-state rules with coupled L2 decay (adamw_coupled_step). */
typedef enum {
  ADAMW_RULE_MOMENTUM = 0, /* s = b*s + g;            p -= lr*s                    */
  ADAMW_RULE_RMSPROP = 1,  /* s = b*s + (1-b)*g*g;    p -= lr*g/(sqrt(s) + eps)    */
  ADAMW_RULE_ADAGRAD = 2   /* s = s + g*g;            p -= lr*g/(sqrt(s) + eps)    */
} adamw_coupled_rule;

/*
 * One step of momentum SGD, RMSprop or Adagrad over every tensor of the plan
 * (fp32 and bf16+remainder modes), with exp_avg as the one state s; exp_avg_sq
 * and exp_avg_slow, if present, are not touched.  "Fix decoupled weight decay
 * ordering in the CUDA Adam/AdEMAMix kernels" (bitsandbytes PR #2040), review
 * of the 1-state kernels: these rules fold the decay into the grad,
 * g = g + p*wd when wd > 0 (coupled L2; a tensor with wd <= 0 gets none), and
 * never decay the parameter directly.  The update formulas are the rules'
 * textbook forms (as torch.optim's SGD with momentum and no dampening,
 * RMSprop without centring, Adagrad without lr decay); no bias correction;
 * the momentum state starting at 0 makes its first step s = g.
 * Float32 sequence, one rounding per operation: g = g_raw [* inv_scale];
 * g = g + p*wd (wd > 0); s' as in the enum above with fl(1-b) for RMSprop;
 * d = s' (momentum) or g / (sqrt(s') + eps); p' = p - lr*d.
 * beta: the momentum or the RMSprop smoothing constant, in [0, 1) (ignored by
 * Adagrad); eps finite and >= 0 (unused by momentum).  20 bytes per element
 * with fp32 params and grads.  lr_dev, step_dev, grad_scale_dev,
 * found_inf_dev, skip and step counting as adamw_step.  EINVAL for an unknown
 * rule, EUNSUPPORTED for 8-bit and 4-bit plans.
 */
adamw_status adamw_coupled_step(adamw_plan* plan, adamw_coupled_rule rule, const float* lr_dev,
                                int32_t* step_dev, float beta, float eps,
                                const float* grad_scale_dev, const float* found_inf_dev,
                                void* stream);

/*
 * The AMP step in one launch ("FusedAdam & PyTorch Lightning AMP": the fused
 * step does the unscale and decides the skip itself): every CTA first scans
 * the raw grads of the elements it owns for +-inf / NaN, the CTAs meet at a
 * grid barrier (a cooperative launch, so all are resident; the wait is bounded
 * at 2 s and reported through adamw_plan_status), and then either all skip --
 * params, states and *step_dev untouched -- or all update, exactly as
 * adamw_check_nonfinite + adamw_step would.  *found_inf_dev (output) receives
 * 1.0f or 0.0f for the caller's loss-scale logic.  On a small plan (see
 * adamw_plan_create) each CTA scans the grads it has staged in shared memory,
 * so they are read from HBM once, and computes its update in place before the
 * vote; only the stores wait for it.  On larger plans the scan reads the grads
 * and the update reads them again (from L2): plans of more than 6 Mi
 * (6,291,456) elements run adamw_check_nonfinite + adamw_step instead, with
 * the same results and the same *found_inf_dev, because past that size the
 * two launches are faster.
 * Other arguments as adamw_step.  fp32 and bf16+remainder modes.
 */
adamw_status adamw_step_amp(adamw_plan* plan, const float* lr_dev, int32_t* step_dev,
                            float beta1, float beta2, float eps,
                            const float* grad_scale_dev, float* found_inf_dev, void* stream);

/*
 * On-device learning-rate schedule: *lr_dev = table[clamp(*step_dev, 0, n-1)],
 * one single-thread launch on `stream`.  Issued before adamw_step on the same
 * stream with the step's own counter, it feeds the step the schedule entry of
 * the step about to run (entry s for the step after s completed steps), so a
 * captured CUDA graph of lookup + step walks a schedule (e.g. the cosine decay
 * of "4 bit Adam should support non constant lr") with no host work per step.
 * table: device fp32 [n], n >= 1; all pointers device, 4-byte aligned.
 */
adamw_status adamw_lr_from_table(const float* table, int32_t n, const int32_t* step_dev,
                                 float* lr_dev, void* stream);

/*
 * Remainder split / join (the rule used by ADAMW_MODE_BF16_REM).
 *   split: a NaN master is first replaced by the quiet NaN 0x7FC00000; then
 *          lo = bits & 0xFFFF; bf16 = (bits >> 16) + (lo >= 0x8000) (mod 2^16);
 *          rem = (int16)lo.  bf16 is the nearest bf16, ties away from zero,
 *          and a NaN for a NaN master (bf16 0x7FC0, remainder 0).
 *   join:  bits = ((bf16 - (rem < 0)) mod 2^16) << 16 | (uint16)rem.
 * join(split(x)) == x for every bit pattern but a NaN, and a NaN for a NaN.
 * Without the replacement the all-ones NaNs (0x7FFF8000..0x7FFFFFFF, the
 * GPU's 0x7FFFFFFF among them, and their negatives) would carry out of the
 * 16-bit half and read as bf16 -0.0 / +0.0.  n >= 0 elements; device
 * pointers, each aligned to its element size.
 */
adamw_status adamw_bf16rem_split(const float* master, uint16_t* bf16, int16_t* rem,
                                 int64_t n, void* stream);
adamw_status adamw_bf16rem_join(const uint16_t* bf16, const int16_t* rem, float* master,
                                int64_t n, void* stream);

/*
 * The default code maps (host arrays of 256 floats, ascending): dynamic
 * exponent maps after Dettmers et al., arXiv:2110.02861 -- after the sign, E
 * zero bits give 10^-E, a one bit, then F fraction bits splitting [0.1, 1]
 * into 2^F equal bins (values at bin centres); signed: E = 0..6, F = 6-E,
 * both signs; unsigned: F = 7-E; each plus exact 0 and +1.0.  Host only.
 */
adamw_status adamw_q8_default_maps(float signed_map[256], float unsigned_map[256]);

/*
 * The Q4 mode's code maps (host arrays of 16 floats, ascending): signed, the
 * dynamic tree above with three magnitude bits (E = 0..2, F = 2-E, both signs,
 * plus 0 and +1.0); unsigned, k/16 for k = 1..16 (no zero: the zero-point
 * problem of "Memory Efficient Optimizers with 4-bit States").  Host only.
 */
adamw_status adamw_q4_default_maps(float signed_map[16], float unsigned_map[16]);

/*
 * Export / import of Q4-mode states (plans in ADAMW_MODE_Q4 only), the 4-bit
 * counterparts of adamw_q8_dequant / adamw_q8_quant: codes are packed
 * [ceil(n/2)] bytes (even element in the low nibble), absmax [ceil(n/128)].
 * dequant: out[i] = map[code(i)] * absmax[i/128].  quant: per 128-element
 * block the absmax of the bit patterns of |x|, then the nearest map entry of
 * x * fl(1/absmax) (both scaled by 2^64 below 2^-64; exact tie -> lower code,
 * NaN -> code 0); an all-zero block stores absmax 0 and the map's zero code
 * (code 0 for the v map, which has no zero).  which: 0 = m map, 1 = v map.
 */
adamw_status adamw_q4_dequant(const adamw_plan* plan, int32_t which, const uint8_t* codes,
                              const float* absmax, float* out, int64_t n, void* stream);
adamw_status adamw_q4_quant(const adamw_plan* plan, int32_t which, const float* x,
                            uint8_t* codes, float* absmax, int64_t n, void* stream);

/* Replace a Q8 plan's maps (host arrays, 256 strictly ascending finite
 * floats each).  Synchronous: waits for all work queued on the device (steps
 * already queued read the old maps), then uploads the new ones.  EUNSUPPORTED
 * if the maps are too dense for the kernel's bucketed nearest-code search. */
adamw_status adamw_q8_set_maps(adamw_plan* plan, const float signed_map[256],
                               const float unsigned_map[256]);

/* Q8 state export / import with a plan's maps, blockwise over n elements
 * (blocks of 256 from element 0).  which: 0 = m (signed map), 1 = v
 * (unsigned map).  dequant: out = map[code] * absmax[block].  quant: absmax
 * and nearest codes as in the step. */
adamw_status adamw_q8_dequant(const adamw_plan* plan, int32_t which, const uint8_t* codes,
                              const float* absmax, float* out, int64_t n, void* stream);
adamw_status adamw_q8_quant(const adamw_plan* plan, int32_t which, const float* x,
                            uint8_t* codes, float* absmax, int64_t n, void* stream);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* adamw_last_error(void);

/* ADAMW_ABI_VERSION of the loaded library. */
int32_t adamw_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ADAMW_GB300_H */
