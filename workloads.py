"""Seeded synthetic inputs for causal kernelized (linear) attention.

This module is shared by the oracle's tests, the CUDA path's parity tests, the
smoke check and the benchmark.  It holds no arithmetic of the method itself:
it only draws Gaussian q, k, v with a fixed seed and rounds them to bf16.

Host recipe (small workloads and all CPU tests):
  * ``rng = numpy.random.default_rng(seed)``;
  * draw q, then k, then v, each ``rng.standard_normal(shape, float32) * sigma``
    (sigma is 1 or 0.5, both exact powers of two, so scaling is exact);
  * for bf16 workloads round each float32 value to bf16 with
    round-to-nearest-even; the same bf16 bits go to the GPU and, widened, to
    the oracle.

Device recipe (the two large workloads, 0.8e9 and 2.4e9 values, which take
minutes to draw on the host): the same draw order and scaling from
``torch.Generator(device).manual_seed(seed)`` (Philox), ``torch.randn`` in
float32, then ``.to(torch.bfloat16)`` (round-to-nearest-even).  The oracle
receives host copies of exactly these bf16 values.

The pages ("Linear attention", learn.pranaymahendrakar.com, Developer
listing; "Linear attention: change the order.", implementation section) use
i.i.d. standard-normal q, k, v; no public dataset or benchmark is involved.
"""
from __future__ import annotations

import dataclasses
from typing import Iterator, Optional, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "causal" | "noncausal" | "decode"
    dtype: str           # "f32" | "bf16"  (dtype of q, k, v, o; states are fp32)
    B: int
    H: int
    N: int               # sequence length (decode: prefill length)
    dk: int
    dv: int
    sigma: float
    seed: int
    chunk: int = 128
    eps: float = 1e-6
    steps: int = 0       # decode only: number of single-token steps

    @property
    def BH(self) -> int:
        return self.B * self.H


# The five workloads the library is specified against.
CAUSAL_F32_SMALL = Workload("causal_f32_b1_h1_n256_d32_c64", "causal", "f32",
                            B=1, H=1, N=256, dk=32, dv=32, sigma=1.0, seed=0, chunk=64)
CAUSAL_BF16 = Workload("causal_bf16_b4_h8_n2048_d64_c128", "causal", "bf16",
                       B=4, H=8, N=2048, dk=64, dv=64, sigma=1.0, seed=1, chunk=128)
NONCAUSAL_BF16 = Workload("noncausal_bf16_b8_h12_n4096_d64", "noncausal", "bf16",
                          B=8, H=12, N=4096, dk=64, dv=64, sigma=1.0, seed=2)
CAUSAL_BF16_LONG = Workload("causal_bf16_b1_h32_n65536_d128_c128", "causal", "bf16",
                            B=1, H=32, N=65536, dk=128, dv=128, sigma=0.5, seed=3, chunk=128)
DECODE_BF16 = Workload("decode_bf16_b128_h32_d128_prefill512_steps1024", "decode", "bf16",
                       B=128, H=32, N=512, dk=128, dv=128, sigma=1.0, seed=4, steps=1024)

ALL = (CAUSAL_F32_SMALL, CAUSAL_BF16, NONCAUSAL_BF16, CAUSAL_BF16_LONG, DECODE_BF16)
BY_NAME = {w.name: w for w in ALL}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round-to-nearest-even); returns uint16 bit patterns.

    Inputs here are finite Gaussian draws, so NaN/Inf handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = u >> np.uint32(16)
    lsb &= np.uint32(1)
    lsb += np.uint32(0x7FFF)
    lsb += u
    lsb >>= np.uint32(16)
    return lsb.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _finish(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def draw_qkv(seed: int, shape_qk: Tuple[int, ...], shape_v: Tuple[int, ...],
             sigma: float, dtype: str,
             rng: Optional[np.random.Generator] = None):
    """Draw q, k (shape_qk) and v (shape_v) in that order from one stream.

    Returns float32 arrays for ``dtype == "f32"`` and uint16 bf16 bit patterns
    for ``dtype == "bf16"``.
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    sig = np.float32(sigma)
    q = rng.standard_normal(shape_qk, dtype=np.float32) * sig
    q = _finish(q, dtype)
    k = rng.standard_normal(shape_qk, dtype=np.float32) * sig
    k = _finish(k, dtype)
    v = rng.standard_normal(shape_v, dtype=np.float32) * sig
    v = _finish(v, dtype)
    return q, k, v


def forward_inputs(w: Workload, N: Optional[int] = None):
    """q, k [B,H,N,dk] and v [B,H,N,dv] for a causal or non-causal workload."""
    n = w.N if N is None else N
    return draw_qkv(w.seed, (w.B, w.H, n, w.dk), (w.B, w.H, n, w.dv), w.sigma, w.dtype)


def decay_gammas(H: int, lo: float = 1e-1, hi: float = 1e-3) -> np.ndarray:
    """Per-head decays for the decayed-state forms: one scalar per head so that
    heads span several timescales, 1 - gamma log-spaced from `lo` (memory of about
    10 tokens, the 0.9 of the fixed-decay exercise) down to `hi` (about 1000
    tokens).  float32 [H]; both the CUDA path and the oracle take these exact values.
    """
    if H == 1:
        return np.array([1.0 - lo], dtype=np.float32)
    return (1.0 - np.logspace(np.log10(lo), np.log10(hi), H)).astype(np.float32)


def random_inputs(seed: int, B: int, H: int, N: int, dk: int, dv: int,
                  dtype: str = "f32", sigma: float = 1.0):
    """Same recipe for arbitrary (test) shapes."""
    return draw_qkv(seed, (B, H, N, dk), (B, H, N, dv), sigma, dtype)


def favor_projection(seed: int, m: int, d: int, dtype: str = "f32", orthogonal: bool = True) -> np.ndarray:
    """Random projections W [m, d] for FAVOR+ features (an input to both sides).

    The Performer draw ("Linear Attention -- Math + Variants", Performer: Gaussian
    rows w_r, made orthogonal to reduce the estimator's variance): blocks of d
    Gaussian rows orthonormalised by a QR factorisation, each row then scaled to
    the length of an independent Gaussian d-vector, so that every row keeps the
    N(0, I) marginal; ceil(m / d) blocks, the first m rows kept.  With
    orthogonal=False the rows are plain N(0, I) draws.  float32, or bf16 bit
    patterns for dtype "bf16" (the rounded values are what both sides use).
    """
    rng = np.random.default_rng(seed)
    if not orthogonal:
        return _finish(rng.standard_normal((m, d)).astype(np.float32), dtype)
    blocks = []
    for _ in range((m + d - 1) // d):
        g = rng.standard_normal((d, d))
        qm, _ = np.linalg.qr(g)
        lengths = np.linalg.norm(rng.standard_normal((d, d)), axis=1)
        blocks.append(qm.T * lengths[:, None])
    return _finish(np.concatenate(blocks, axis=0)[:m].astype(np.float32), dtype)


class DecodeInputs:
    """Decode workload: a causal prefill of ``w.N`` tokens, then ``w.steps`` steps.

    Draw order from ``default_rng(w.seed)``: prefill q, k, v [B,H,N,d], then
    decode q, k, v [steps,B,H,d] (q entirely, then k, then v).  Decode slices
    are produced in step order without materialising whole float32 arrays;
    chunked draws of one stream reproduce the single large draw exactly.
    """

    def __init__(self, w: Workload, steps: Optional[int] = None):
        self.w = w
        self.steps = w.steps if steps is None else steps

    def prefill(self):
        w = self.w
        rng = np.random.default_rng(w.seed)
        q, k, v = draw_qkv(w.seed, (w.B, w.H, w.N, w.dk), (w.B, w.H, w.N, w.dv),
                           w.sigma, w.dtype, rng=rng)
        return q, k, v, rng

    def decode_all(self, slice_steps: int = 64):
        """All decode-step inputs: q,k [steps,B,H,dk], v [steps,B,H,dv].

        The stream always covers the full ``w.steps`` so that a shorter
        ``steps`` gives a prefix of the same inputs.
        """
        w = self.w
        _, _, _, rng = self.prefill()
        sig = np.float32(w.sigma)
        out = []
        for d in (w.dk, w.dk, w.dv):
            dt = np.uint16 if w.dtype == "bf16" else np.float32
            arr = np.empty((self.steps, w.B, w.H, d), dtype=dt)
            s = 0
            while s < w.steps:
                n = min(slice_steps, w.steps - s)
                x = rng.standard_normal((n, w.B, w.H, d), dtype=np.float32) * sig
                lo, hi = s, min(s + n, self.steps)
                if lo < hi:
                    arr[lo:hi] = _finish(x[: hi - lo], w.dtype)
                s += n
            out.append(arr)
        return tuple(out)


def iter_heads(BH: int, group: int) -> Iterator[Tuple[int, int]]:
    for s in range(0, BH, group):
        yield s, min(BH, s + group)


# ---------------------------------------------------------------------------
# Device recipe (torch, Philox) for the large workloads.
# ---------------------------------------------------------------------------
def _torch_dtype(dtype: str):
    import torch
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def _device_draw(gen, shape, sigma, dtype, device):
    import torch
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(_torch_dtype(dtype))


def device_forward_inputs(w: Workload, device: str = "cuda"):
    """q, k [B,H,N,dk], v [B,H,N,dv] as torch tensors drawn on ``device``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    q = _device_draw(g, (w.B, w.H, w.N, w.dk), w.sigma, w.dtype, device)
    k = _device_draw(g, (w.B, w.H, w.N, w.dk), w.sigma, w.dtype, device)
    v = _device_draw(g, (w.B, w.H, w.N, w.dv), w.sigma, w.dtype, device)
    return q, k, v


def device_decode_inputs(w: Workload, device: str = "cuda"):
    """Prefill q,k,v [B,H,N,d] then decode q,k,v [steps,B,H,d], drawn on ``device``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    pre = tuple(_device_draw(g, (w.B, w.H, w.N, d), w.sigma, w.dtype, device) for d in (w.dk, w.dk, w.dv))
    dec = tuple(_device_draw(g, (w.steps, w.B, w.H, d), w.sigma, w.dtype, device) for d in (w.dk, w.dk, w.dv))
    return pre, dec


def to_host_bits(t) -> np.ndarray:
    """Host copy of a device tensor in the oracle's input form (bf16 bits or float32)."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy().astype(np.float32)
