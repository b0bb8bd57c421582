"""Fused AdamW optimizer step for GB300 (sm_103a) behind a C ABI (libadamw).

``_capi`` mirrors ``include/adamw.h`` one function per entry point.
``FusedAdamW`` is the same calls with torch tensors in place of raw pointers:
it checks dtypes, devices and contiguity, builds the ``adamw_tensor`` list
and keeps the tensors alive for the plan's lifetime.  Every step of the
update runs in the library's CUDA kernels; there is no CPU fallback -- if the
library is missing, importing ``_capi``'s functions raises.
"""

from __future__ import annotations

from . import _capi
from ._capi import (  # noqa: F401
    AdamWError, adamw_abi_version, adamw_ademamix_step, adamw_bf16rem_join, adamw_bf16rem_split,
    adamw_coupled_step, adamw_lion_step, adamw_mini_plan_create, adamw_mini_step,
    adamw_q4_default_maps,
    adamw_check_nonfinite, adamw_last_error, adamw_lr_from_table, adamw_plan_create,
    adamw_plan_destroy,
    adamw_plan_info, adamw_plan_status, adamw_q8_default_maps, adamw_q8_dequant, adamw_q8_quant,
    adamw_q8_set_maps, adamw_step, adamw_step_amp, adamw_step_noalloc, adamw_step_noalloc_status,
    adamw_wait_selftest,
)

MODES = {"fp32": _capi.MODE_FP32, "bf16_rem": _capi.MODE_BF16_REM, "q8": _capi.MODE_Q8,
         "q4": _capi.MODE_Q4}


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else stream


def _grad_dtype(dt) -> int:
    import torch
    table = {torch.float32: _capi.F32, torch.float16: _capi.F16, torch.bfloat16: _capi.BF16}
    if dt not in table:
        raise TypeError(f"unsupported grad dtype {dt}")
    return table[dt]


class FusedAdamW:
    """A plan over a fixed list of tensors; ``step`` is one launch of ``adamw_step``.

    mode "fp32":     params, exp_avgs, exp_avg_sqs float32.
    mode "bf16_rem": params bfloat16 + ``param_rems`` int16; states float32.
    mode "q8":       params float32; exp_avgs / exp_avg_sqs uint8 codes plus
                     ``absmax_m`` / ``absmax_v`` float32 [ceil(numel/256)].
    mode "q4":       params float32; exp_avgs / exp_avg_sqs uint8 [ceil(numel/2)],
                     two 4-bit codes per byte; absmax float32 [ceil(numel/128)].
    Grads: float32, float16 or bfloat16, one dtype for the whole list.
    ``weight_decays``: one float per tensor.
    ``exp_avg_sqs=None`` (fp32 / bf16_rem only) makes a plan for the 1-state
    steps ``step_lion`` and ``step_coupled`` alone.
    ``v_blocks`` (fp32 / bf16_rem): one Adam-mini block length per tensor; the
    tensor's exp_avg_sq then holds numel / block values and the plan steps with
    ``step_mini``.
    """

    def __init__(self, params, grads, exp_avgs, exp_avg_sqs, weight_decays, *, mode="fp32",
                 param_rems=None, absmax_m=None, absmax_v=None, exp_avg_slows=None, v_blocks=None):
        import torch
        if mode not in MODES:
            raise ValueError(f"mode must be one of {sorted(MODES)}")
        n = len(params)
        if exp_avg_sqs is None:
            exp_avg_sqs = [None] * n
        lists = [grads, exp_avgs, exp_avg_sqs, weight_decays]
        if any(len(x) != n for x in lists):
            raise ValueError("all lists must have one entry per param")
        self.mode = mode
        rems = param_rems if param_rems is not None else [None] * n
        ams = absmax_m if absmax_m is not None else [None] * n
        avs = absmax_v if absmax_v is not None else [None] * n
        slows = exp_avg_slows if exp_avg_slows is not None else [None] * n
        pdt = torch.bfloat16 if mode == "bf16_rem" else torch.float32
        sdt = torch.uint8 if mode in ("q8", "q4") else torch.float32
        gdt = grads[0].dtype if n else torch.float32
        recs = []
        for i in range(n):
            p, g, m, v = params[i], grads[i], exp_avgs[i], exp_avg_sqs[i]
            for name, t, dt in (("param", p, pdt), ("exp_avg", m, sdt), ("exp_avg_sq", v, sdt),
                                ("grad", g, gdt)):
                if t is None and name == "exp_avg_sq":
                    continue
                if t.dtype != dt:
                    raise TypeError(f"tensor {i}: {name} must be {dt}, got {t.dtype}")
                if not t.is_contiguous() or t.device.type != "cuda":
                    raise ValueError(f"tensor {i}: {name} must be a contiguous CUDA tensor")
                want = (p.numel() + 1) // 2 if (mode == "q4" and name in ("exp_avg", "exp_avg_sq")) \
                    else p.numel()
                if v_blocks is not None and name == "exp_avg_sq":
                    want = p.numel() // max(1, int(v_blocks[i]))
                if t.numel() != want:
                    raise ValueError(f"tensor {i}: {name} has {t.numel()} elements, expected {want}")
            if mode == "bf16_rem" and (rems[i] is None or rems[i].dtype != torch.int16
                                       or rems[i].numel() != p.numel()):
                raise TypeError(f"tensor {i}: bf16_rem mode needs an int16 remainder per element")
            if mode in ("q8", "q4"):
                blk = _capi.Q8_BLOCK if mode == "q8" else _capi.Q4_BLOCK
                nb = (p.numel() + blk - 1) // blk
                for name, a in (("absmax_m", ams[i]), ("absmax_v", avs[i])):
                    if a is None or a.dtype != torch.float32 or a.numel() < nb:
                        raise TypeError(f"tensor {i}: {mode} mode needs {name} float32 [{nb}]")
            if slows[i] is not None and (slows[i].dtype != torch.float32
                                         or slows[i].numel() != p.numel()):
                raise TypeError(f"tensor {i}: exp_avg_slow must be float32 with one entry per element")
            recs.append(_capi.adamw_tensor(
                _ptr(p), _ptr(rems[i]), _ptr(g), _ptr(m), _ptr(v), _ptr(ams[i]), _ptr(avs[i]),
                int(p.numel()), float(weight_decays[i]), _ptr(slows[i])))
        self._keep = (list(params), list(grads), list(exp_avgs), list(exp_avg_sqs), rems, ams, avs,
                      slows)
        if v_blocks is not None:
            if len(v_blocks) != n:
                raise ValueError("v_blocks must have one entry per param")
            self.plan = adamw_mini_plan_create(recs, [int(b) for b in v_blocks], MODES[mode],
                                               _grad_dtype(gdt))
        else:
            self.plan = adamw_plan_create(recs, MODES[mode], _grad_dtype(gdt))

    def info(self) -> dict:
        return adamw_plan_info(self.plan)

    def status(self) -> int:
        """Device-side fault bits (0 = healthy); raises AdamWError if a bounded wait gave up."""
        return adamw_plan_status(self.plan)

    def check_nonfinite(self, found_inf, stream=None) -> None:
        adamw_check_nonfinite(self.plan, _ptr(found_inf), _stream(stream))

    def step(self, lr, step, *, betas=(0.9, 0.999), eps=1e-8, grad_scale=None, found_inf=None,
             stream=None) -> None:
        """lr: float32 CUDA scalar tensor; step: int32 CUDA scalar (completed steps)."""
        adamw_step(self.plan, _ptr(lr), _ptr(step), float(betas[0]), float(betas[1]), float(eps),
                   _ptr(grad_scale), _ptr(found_inf), _stream(stream))

    def step_ademamix(self, lr, step, *, betas=(0.9, 0.999, 0.9999), alpha=5.0, eps=1e-8,
                      grad_scale=None, found_inf=None, stream=None) -> None:
        """AdEMAMix step (the plan needs exp_avg_slows); betas = (b1, b2, b3)."""
        adamw_ademamix_step(self.plan, _ptr(lr), _ptr(step), float(betas[0]), float(betas[1]),
                            float(betas[2]), float(alpha), float(eps), _ptr(grad_scale),
                            _ptr(found_inf), _stream(stream))

    def step_mini(self, lr, step, *, betas=(0.9, 0.999), eps=1e-8, grad_scale=None, found_inf=None,
                  stream=None) -> None:
        """Adam-mini step (plans made with ``v_blocks``)."""
        adamw_mini_step(self.plan, _ptr(lr), _ptr(step), float(betas[0]), float(betas[1]),
                        float(eps), _ptr(grad_scale), _ptr(found_inf), _stream(stream))

    def step_lion(self, lr, step, *, betas=(0.9, 0.99), grad_scale=None, found_inf=None,
                  stream=None) -> None:
        """Lion step (decay, then a step of lr against sign(b1*m + (1-b1)*g));
        betas = (b1, b2); exp_avg_sqs are not touched."""
        adamw_lion_step(self.plan, _ptr(lr), _ptr(step), float(betas[0]), float(betas[1]),
                        _ptr(grad_scale), _ptr(found_inf), _stream(stream))

    def step_coupled(self, rule, lr, step, *, beta=0.9, eps=1e-8, grad_scale=None, found_inf=None,
                     stream=None) -> None:
        """Momentum SGD, RMSprop or Adagrad (``rule``) with coupled L2 decay;
        exp_avgs hold the one state, exp_avg_sqs are not touched."""
        adamw_coupled_step(self.plan, _capi.RULES[rule], _ptr(lr), _ptr(step), float(beta),
                           float(eps), _ptr(grad_scale), _ptr(found_inf), _stream(stream))

    def step_amp(self, lr, step, found_inf, *, betas=(0.9, 0.999), eps=1e-8, grad_scale=None,
                 stream=None) -> None:
        """Check + step in one launch; found_inf (float32 CUDA scalar) is written, not read."""
        adamw_step_amp(self.plan, _ptr(lr), _ptr(step), float(betas[0]), float(betas[1]),
                       float(eps), _ptr(grad_scale), _ptr(found_inf), _stream(stream))

    def set_maps(self, signed_map, unsigned_map) -> None:
        adamw_q8_set_maps(self.plan, signed_map, unsigned_map)

    def close(self) -> None:
        if getattr(self, "plan", None):
            adamw_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
