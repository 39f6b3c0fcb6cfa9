"""Helpers for the GPU parity tests: host<->device marshalling and error metrics.

Tolerances (written where they are asserted):
  fp32 inputs: normwise max|gpu - oracle| / max|oracle| <= 1e-5 over the whole
               output (elementwise relative error is ill-conditioned where o ~ 0);
  bf16 inputs: max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3.
"""
from __future__ import annotations

import numpy as np

import workloads

F32_NORMWISE = 1e-5
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3


def to_dev(x: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        assert x.dtype == np.uint16
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def from_dev(t) -> np.ndarray:
    """Device tensor (fp32 or bf16) -> float64 numpy."""
    import torch
    if t.dtype == torch.bfloat16:
        bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return workloads.bf16_bits_to_f32(bits).astype(np.float64)
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray) -> dict:
    d = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    return {
        "max_abs": float(d.max()) if d.size else 0.0,
        "mean_abs": float(d.mean()) if d.size else 0.0,
        "normwise": float(d.max() / scale) if d.size and scale > 0 else 0.0,
        "finite": bool(np.all(np.isfinite(got))),
    }


def assert_parity(got, ref, dtype: str, what: str = ""):
    e = errors(got, ref)
    assert e["finite"], (what, "non-finite output")
    if dtype == "f32":
        assert e["normwise"] <= F32_NORMWISE, (what, e)
    else:
        assert e["max_abs"] <= BF16_MAX_ABS and e["mean_abs"] <= BF16_MEAN_ABS, (what, e)
    return e
