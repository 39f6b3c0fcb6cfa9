"""FAVOR+ features and linear attention on them, GPU vs the float64 oracle.

"Linear Attention -- Math + Variants", Performer: phi(x)_r = exp(w_r . x -
|x|^2 / 2) / sqrt(m) with Gaussian (here orthogonal-block) projections w_r, the
features then used in place of elu + 1 by the causal and non-causal forms.
Every call goes through the C ABI; the projections come from
``workloads.favor_projection`` and reach both sides as the same values.

Inputs are drawn at sigma = 0.5 (the Performer's usual d^(-1/4) input scaling is
about 0.35 at d = 64), so that w_r . x - |x|^2 / 2 stays within fp32's exponent
range at d = 128: the features are then compared elementwise, relatively.

Tolerances:
  features, fp32: |gpu - oracle| / oracle <= 1e-4.  The exponent w_r . x - |x|^2 / 2
    (|.| up to about 60 here) carries the rounding of two fp32 dot products of d
    <= 128 terms, a few 1e-6 in practice (the worst-case bound d * 2^-24 * sum of
    |terms| is about 1e-3); the exponential adds a few ulps;
  features, bf16: <= 2^-8: the output's own rounding (2^-9) plus the exponent's
    fp32 error;
  attention: the bounds of the other forward tests (fp32 normwise 1e-5; bf16 max
    abs 2e-2, mean abs 2e-3): normalised outputs stay weighted averages of v.
"""
import numpy as np
import pytest

import workloads
from gpu_util import assert_parity, from_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SIGMA = 0.5
FEATURE_RTOL = {"f32": 1e-4, "bf16": 2.0 ** -8}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_kernelized_attention_gb300 import build
    build.build()
    import causal_kernelized_attention_gb300 as la
    la.load_library()
    return la


def la():
    import causal_kernelized_attention_gb300 as m
    return m


def widen(x, dtype):
    """The values an array holds (bf16 bit patterns or fp32), as float64."""
    return workloads.bf16_bits_to_f32(x).astype(np.float64) if dtype == "bf16" else np.asarray(x, np.float64)


def inputs(seed, B, H, N, d, dv, m, dtype):
    q, k, v = workloads.random_inputs(seed, B, H, N, d, dv, dtype, sigma=SIGMA)
    w = workloads.favor_projection(seed + 1, m, d, dtype)
    return q, k, v, w


@pytest.mark.parametrize("dtype,B,H,N,d,m", [
    ("bf16", 2, 3, 300, 64, 64), ("bf16", 2, 3, 300, 64, 128), ("bf16", 1, 2, 1000, 128, 64),
    ("bf16", 1, 2, 1000, 128, 128), ("bf16", 1, 1, 1, 64, 64), ("bf16", 3, 1, 129, 128, 128),
    ("bf16", 2, 3, 257, 32, 64), ("bf16", 1, 2, 200, 64, 32),
    ("f32", 2, 3, 300, 64, 128), ("f32", 1, 2, 129, 128, 32), ("f32", 1, 1, 1, 32, 32),
])
def test_features(orc, dtype, B, H, N, d, m):
    """Tensor-core shapes (bf16, d and m in {64, 128}, N >= 128; ragged tiles) and
    CUDA-core shapes (a single row, d or m = 32, fp32)."""
    x, _, _, w = inputs(21000 + N + d + m, B, H, N, d, d, m, dtype)
    phi = la().la_favor_features(to_dev(x, dtype), to_dev(w, dtype))
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.favor_features(x, widen(w, dtype))
    got = from_dev(phi)
    assert got.shape == ref.shape == (B, H, N, m)
    assert np.all(np.isfinite(got)) and np.all(ref > 0)
    rel = np.abs(got - ref) / ref
    assert rel.max() <= FEATURE_RTOL[dtype], (dtype, d, m, float(rel.max()))


@pytest.mark.parametrize("dtype,B,H,N,d,dv,m,chunk", [
    ("bf16", 2, 3, 300, 64, 64, 64, 128), ("bf16", 1, 4, 1000, 128, 128, 128, 128),
    ("bf16", 2, 2, 2000, 64, 128, 128, 128), ("bf16", 1, 2, 20000, 64, 64, 64, 128),
    ("bf16", 2, 3, 257, 128, 64, 64, 128), ("bf16", 2, 3, 300, 64, 32, 64, 128),
    ("bf16", 2, 3, 300, 32, 64, 64, 64), ("bf16", 4, 8, 2048, 64, 64, 64, 128),
    ("f32", 2, 3, 300, 64, 64, 64, 128), ("f32", 1, 2, 129, 32, 32, 128, 64),
])
def test_causal_favor(orc, dtype, B, H, N, d, dv, m, chunk):
    """Tensor-core attention (bf16, m = dv in {64, 128}: short and scan modes, the
    B=4 H=8 N=2048 d=64 headline shape) and CUDA-core shapes (m != dv, chunk 64, fp32)."""
    q, k, v, w = inputs(22000 + N + d + dv + m, B, H, N, d, dv, m, dtype)
    o = la().la_forward_causal_favor(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), to_dev(w, dtype),
                                     chunk=chunk)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.causal_favor(q, k, v, widen(w, dtype))
    assert_parity(from_dev(o), ref, dtype, ("causal_favor", N, d, dv, m))


@pytest.mark.parametrize("dtype,B,H,N,d,dv,m", [
    ("bf16", 2, 3, 1000, 64, 64, 64), ("bf16", 1, 4, 3000, 128, 128, 128), ("bf16", 2, 2, 500, 64, 128, 128),
    ("bf16", 2, 3, 300, 64, 32, 128), ("f32", 2, 3, 300, 64, 64, 64),
    ("bf16", 8, 12, 4096, 64, 64, 64),  # the benchmark's FAVOR+ non-causal workload
    # d = m = 64 computes the features inside the attention kernel: one chunk, ragged
    # tails, many one-chunk heads, several key splits per head, dv = 32
    ("bf16", 2, 3, 128, 64, 64, 64), ("bf16", 2, 3, 129, 64, 64, 64), ("bf16", 64, 16, 128, 64, 64, 64),
    ("bf16", 4, 40, 4173, 64, 64, 64), ("bf16", 2, 3, 1000, 64, 32, 64), ("bf16", 1, 2, 20000, 64, 64, 64),
])
def test_noncausal_favor(orc, dtype, B, H, N, d, dv, m):
    q, k, v, w = inputs(23000 + N + d + dv + m, B, H, N, d, dv, m, dtype)
    o = la().la_forward_noncausal_favor(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), to_dev(w, dtype))
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.noncausal_favor(q, k, v, widen(w, dtype))
    assert_parity(from_dev(o), ref, dtype, ("noncausal_favor", N, d, dv, m))


def normwise(got, ref):
    return float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))


# States (normwise): the unnormalised sums keep the features' own error, which the
# features test bounds elementwise -- fp32: the exponent's rounding, a few 1e-6 relative
# on the largest features that dominate S (bound 1e-4, the features' bound); bf16: the
# features' single rounding, 2^-9 relative (bound 1e-2).
STATE_TOL = {"f32": 1e-4, "bf16": 1e-2}


@pytest.mark.parametrize("dtype,B,H,N,d,dv,m", [
    ("bf16", 2, 3, 300, 64, 64, 64), ("bf16", 1, 4, 1000, 128, 128, 128), ("bf16", 2, 3, 257, 64, 32, 128),
    ("bf16", 2, 2, 100, 128, 64, 64), ("f32", 2, 3, 300, 64, 64, 64), ("f32", 1, 2, 129, 32, 128, 32),
])
def test_prefill_state_favor(orc, dtype, B, H, N, d, dv, m):
    """S = sum_t phi(k_t) v_t^T, z = sum_t phi(k_t) on FAVOR+ features: tensor-core state
    (bf16, m = dv in {64, 128}, N >= 128) and CUDA-core shapes."""
    _, k, v, w = inputs(25000 + N + d + dv + m, B, H, N, d, dv, m, dtype)
    S, z = la().la_prefill_state_favor(to_dev(k, dtype), to_dev(v, dtype), to_dev(w, dtype))
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    Sr, zr = orc.prefill_state_general(orc.favor_features(k, widen(w, dtype)), widen(v, dtype), fmap="identity",
                                       shift=0.0)
    assert normwise(from_dev(S), Sr) <= STATE_TOL[dtype], ("S", dtype, N, d, dv, m)
    assert normwise(from_dev(z), zr) <= STATE_TOL[dtype], ("z", dtype, N, d, dv, m)


def test_prefill_state_favor_empty_sequence_writes_zeros():
    kd = torch.empty((2, 3, 0, 64), dtype=torch.bfloat16, device="cuda")
    w = to_dev(workloads.favor_projection(25900, 64, 64, "bf16"), "bf16")
    S = torch.full((2, 3, 64, 64), 7.0, device="cuda")
    z = torch.full((2, 3, 64), 7.0, device="cuda")
    la().la_prefill_state_favor(kd, kd, w, S, z)
    torch.cuda.synchronize()
    assert torch.all(S == 0) and torch.all(z == 0)


@pytest.mark.parametrize("dtype,B,H,d,dv,m", [
    ("bf16", 32, 4, 64, 64, 64), ("bf16", 16, 8, 128, 128, 128), ("bf16", 2, 3, 64, 32, 128),
    ("f32", 2, 3, 64, 64, 64), ("f32", 32, 4, 32, 64, 32),
])
def test_decode_step_favor(orc, dtype, B, H, d, dv, m):
    """A 64-token FAVOR+ prefill, then 4 decode steps: each step's o and the final S, z
    against the oracle's decode steps on the oracle's features (B*H >= 128 rows take the
    tensor-core features kernel for bf16 with d, m in {64, 128})."""
    N, steps = 64, 4
    _, kp, vp, w = inputs(26000 + d + dv + m + B, B, H, N, d, dv, m, dtype)
    q, k, v = workloads.random_inputs(26500 + d + m + B, steps, B, H, d, dv, dtype, sigma=SIGMA)
    wd = to_dev(w, dtype)
    S, z = la().la_prefill_state_favor(to_dev(kp, dtype), to_dev(vp, dtype), wd)
    wr = widen(w, dtype)
    Sr, zr = orc.prefill_state_general(orc.favor_features(kp, wr), widen(vp, dtype), fmap="identity", shift=0.0)
    Sr, zr = np.ascontiguousarray(Sr), np.ascontiguousarray(zr)
    for t in range(steps):
        o = la().la_decode_step_favor(S, z, to_dev(q[t], dtype), to_dev(k[t], dtype), to_dev(v[t], dtype), wd)
        torch.cuda.synchronize()
        ref = orc.decode_step_general(Sr, zr, orc.favor_features(q[t], wr), orc.favor_features(k[t], wr),
                                      widen(v[t], dtype), fmap="identity", shift=0.0, normalize=True)
        assert_parity(from_dev(o), ref, dtype, ("decode_favor", t, d, dv, m))
    assert la().la_get_device_status() == 0
    assert normwise(from_dev(S), Sr) <= STATE_TOL[dtype]
    assert normwise(from_dev(z), zr) <= STATE_TOL[dtype]


def test_causal_favor_first_row_and_graph_replay(orc):
    """o_0 = v_0 (one key) and a captured CUDA graph of the two-launch call gives
    the same output as the eager call (scratch allocated stream-ordered inside)."""
    dtype, B, H, N, d = "bf16", 2, 4, 1024, 64
    q, k, v, w = inputs(24000, B, H, N, d, d, d, dtype)
    qd, kd, vd, wd = (to_dev(t, dtype) for t in (q, k, v, w))
    eager = la().la_forward_causal_favor(qd, kd, vd, wd)
    torch.cuda.synchronize()
    o0 = from_dev(eager)[:, :, 0, :]
    assert np.max(np.abs(o0 - widen(v, dtype)[:, :, 0, :])) <= 2e-2
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        la().la_forward_causal_favor(qd, kd, vd, wd, o=out, stream=s)  # warm the pools outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            la().la_forward_causal_favor(qd, kd, vd, wd, o=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    assert torch.equal(out, eager)


def test_noncausal_favor_features_in_the_attention_kernel():
    """bf16 with d = m = 64: one launch of the non-causal kernel, no separate
    features kernel (a profiler pass over one call)."""
    from torch.profiler import ProfilerActivity, profile
    B, H, N, d = 2, 3, 1000, 64
    gen = torch.Generator(device="cuda").manual_seed(3)
    q, k, v = [(0.5 * torch.randn((B, H, N, d), device="cuda", generator=gen)).to(torch.bfloat16) for _ in range(3)]
    w = torch.randn((d, d), device="cuda", generator=gen).to(torch.bfloat16)
    call = lambda: la().la_forward_noncausal_favor(q, k, v, w)
    call()
    torch.cuda.synchronize()
    names = []
    for _ in range(2):  # a first profiler session can come back empty
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            call()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
        if names:
            break
    if not names:
        pytest.skip("the profiler recorded no kernels")
    assert any("noncausal_tc_kernel" in n for n in names), names
    assert not any("favor_tc_kernel" in n for n in names), names
