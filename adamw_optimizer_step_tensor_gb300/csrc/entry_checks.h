// entry_checks.h -- argument checks and launch-argument setup shared by the
// extern "C" step entry points (capi.cpp, noalloc.cu).  Host code only.
#pragma once

#include "internal.h"

namespace adamw {

// A non-OK status has set the adamw_last_error() message (capi.cpp).
adamw_status check_mode_dtype(int mode, int grad_dtype);   // EDTYPE for unknown values
adamw_status check_step_scalars(const float* lr_dev, const int32_t* step_dev,
                                const float* grad_scale_dev, const float* found_inf_dev,
                                float beta1, float beta2);
adamw_status check_eps(float eps);

// The launch arguments every step shares; rule-specific fields keep their
// neutral values (no slow EMA, no code maps, no Adam-mini blocks).
inline StepArgs base_step_args(const TensorDesc* tensors, const Chunk* chunks, int64_t n_chunks,
                               StepScratch* scratch, const float* lr_dev, int32_t* step_dev,
                               const float* grad_scale_dev, const float* found_inf_dev,
                               float beta1, float beta2, float eps) {
  StepArgs a;
  a.tensors = tensors;
  a.chunks = chunks;
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
  a.scratch = scratch;
  a.qt = nullptr;
  a.refine = 1;
  return a;
}

}  // namespace adamw
