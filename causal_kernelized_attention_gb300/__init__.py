"""Causal kernelized (linear) attention, phi = elu + 1, on GB300 (sm_103a).

Thin Python binding over the C ABI of ``liblinattn.so`` (declared in
``include/la.h``).  Every function below only checks and marshals arguments
(device pointers, sizes, the current CUDA stream) and calls the C entry point
of the same name; all arithmetic runs in the library's CUDA kernels.  There is
no CPU or PyTorch fallback: if the library is missing or fails to load, the
import of this package's functions raises.

Tensors are PyTorch CUDA tensors (PyTorch supplies device memory and streams):
  q, k [B, H, N, dk], v, o [B, H, N, dv], fp32 or bf16, contiguous;
  decode: q, k [B, H, dk], v, o [B, H, dv]; S [B, H, dk, dv] and z [B, H, dk] fp32;
  decayed forms: gamma [H] fp32, one decay per head;
  gated forms: alpha fp32 shaped like k, one gate per (token, key feature);
  *_ex forms: feature_map "elu1" | "relu" (max(x, 0) + shift) | "identity" (x + shift),
  normalize True | False, and an optional gamma;
  FAVOR+ forms: projections w [m, d] of the inputs' dtype, features [B, H, N, m].
"""
from __future__ import annotations

from ._binding import (LA_BF16, LA_F32, LA_PHI_ELU1, LA_PHI_IDENTITY, LA_PHI_RELU, LAError, Variant, lib_path,
                       la_backward_causal, la_favor_features, la_forward_causal_favor, la_forward_noncausal_favor,
                       la_prefill_state_favor, la_decode_step_favor, la_decode_step, la_decode_step_decay, la_decode_step_ex, la_forward_causal,
                       la_forward_causal_decay, la_forward_causal_ex, la_forward_noncausal, la_forward_noncausal_ex,
                       la_prefill_state_ex, la_forward_noncausal_noalloc, la_get_device_status, la_kernel_launches, la_last_cuda_error,
                       la_prefill_state, la_prefill_state_decay, la_status_string, la_version, load_library,
                       la_forward_causal_gated, la_prefill_state_gated, la_decode_step_gated)

__all__ = [
    "LA_BF16", "LA_F32", "LA_PHI_ELU1", "LA_PHI_IDENTITY", "LA_PHI_RELU", "LAError", "Variant", "lib_path",
    "la_backward_causal", "la_favor_features", "la_forward_causal_favor", "la_forward_noncausal_favor",
    "la_prefill_state_favor", "la_decode_step_favor",
    "la_decode_step", "la_decode_step_decay", "la_decode_step_ex", "la_forward_causal", "la_forward_causal_decay",
    "la_forward_causal_ex", "la_forward_noncausal_ex", "la_prefill_state_ex",
    "la_forward_noncausal", "la_forward_noncausal_noalloc", "la_get_device_status", "la_kernel_launches", "la_last_cuda_error", "la_prefill_state",
    "la_prefill_state_decay", "la_forward_causal_gated", "la_prefill_state_gated", "la_decode_step_gated",
    "la_status_string", "la_version", "load_library",
]
