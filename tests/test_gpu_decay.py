"""Decayed-state forms on the GPU vs the float64 oracle ("Linear Attention --
Math + Variants", RetNet and gated linear attention: S_i = g S_{i-1} +
phi(k_i) v_i^T with one scalar g per head; the normaliser z decays with the
same g).  Every call goes through the C ABI.  Tolerances as the undecayed
parity tests: fp32 normwise 1e-5; bf16 max abs 2e-2, mean abs 2e-3.
"""
import numpy as np
import pytest

import workloads
from gpu_util import assert_parity, errors, from_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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


def run_decay(q, k, v, gamma, dtype, chunk, eps=1e-6):
    g = torch.from_numpy(np.ascontiguousarray(gamma, dtype=np.float32)).cuda()
    o = la().la_forward_causal_decay(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), g,
                                     chunk=chunk, eps=eps)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    return from_dev(o)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,dk,dv,chunk", [
    (1, 32, 32, 64), (63, 64, 64, 64), (65, 64, 64, 64), (129, 128, 128, 128), (300, 64, 64, 128),
    (257, 64, 128, 64), (130, 128, 32, 128), (1000, 128, 128, 128), (2000, 32, 64, 64),
])
def test_causal_decay_cases(orc, dtype, N, dk, dv, chunk):
    """Three heads with decays 0.9, 0.99, 0.999: ragged last chunks, one and many chunks."""
    B, H = 2, 3
    q, k, v = workloads.random_inputs(7000 + N + dk + dv, B, H, N, dk, dv, dtype)
    gamma = workloads.decay_gammas(H)
    got = run_decay(q, k, v, gamma, dtype, chunk)
    ref = orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64))
    assert_parity(got, ref, dtype, (N, dk, dv, chunk))


@pytest.mark.parametrize("chunk", [64, 128])
def test_causal_decay_special_gammas(orc, chunk):
    """g = 1 is the undecayed causal form; g = 0 returns v_i; g = 1/2 is exact in
    fp32 (its powers are powers of two)."""
    B, H, N, d = 2, 3, 333, 64
    q, k, v = workloads.random_inputs(8123 + chunk, B, H, N, d, d, "f32")
    gamma = np.array([1.0, 0.0, 0.5], dtype=np.float32)
    got = run_decay(q, k, v, gamma, "f32", chunk)
    ref = orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64))
    assert_parity(got, ref, "f32", "special gammas")
    assert_parity(got[:, 0], orc.causal_recurrent(q, k, v)[:, 0], "f32", "g = 1")
    np.testing.assert_allclose(got[:, 1], v[:, 1].astype(np.float64), rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("B,H,N,d", [
    (1, 1, 128, 64), (1, 1, 128, 128), (2, 3, 129, 64), (1, 2, 255, 128), (3, 2, 1000, 64),
    (2, 3, 2000, 128), (4, 8, 2048, 64), (1, 3, 20000, 64), (1, 2, 20000, 128),
])
def test_causal_decay_tensor_core_shapes(orc, B, H, N, d):
    """Shapes of the tensor-core path (bf16, dk = dv in {64, 128}, chunk 128):
    ragged last chunks, short sequences split into segments that sum their own
    decayed prefix, and long sequences whose segments combine decayed
    aggregates by look-back."""
    q, k, v = workloads.random_inputs(12000 + N + d, B, H, N, d, d, "bf16")
    gamma = workloads.decay_gammas(H)
    got = run_decay(q, k, v, gamma, "bf16", 128)
    ref = orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64))
    e = assert_parity(got, ref, "bf16", (B, H, N, d))
    assert e["normwise"] < 2e-2, e


@pytest.mark.parametrize("B,N,d", [(2, 1000, 64), (1, 3000, 128), (1, 20000, 64)])
def test_causal_decay_tensor_core_special_gammas(orc, B, N, d):
    """g = 0 (o_i = v_i), 1/2, 1 (the undecayed form) and 0.999 on the tensor-core path."""
    H = 4
    q, k, v = workloads.random_inputs(13000 + N + d, B, H, N, d, d, "bf16")
    gamma = np.array([0.0, 0.5, 1.0, 0.999], dtype=np.float32)
    got = run_decay(q, k, v, gamma, "bf16", 128)
    ref = orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64))
    assert_parity(got, ref, "bf16", (B, N, d))
    assert_parity(got[:, 2], orc.causal_recurrent(q, k, v)[:, 2], "bf16", "g = 1")
    vv = workloads.bf16_bits_to_f32(v[:, 0]).astype(np.float64)
    assert np.max(np.abs(got[:, 0] - vv)) <= 2e-2


def test_causal_decay_gamma_one_matches_undecayed_tensor_core():
    """g = 1 on the tensor-core path gives the undecayed kernel's result (every
    weight is exactly 1; D = 128 accumulates O in another order)."""
    for d in (64, 128):
        gen = torch.Generator(device="cuda").manual_seed(21 + d)
        q, k, v = ((torch.randn((2, 4, 3000, d), device="cuda", generator=gen) * 0.5).to(torch.bfloat16)
                   for _ in range(3))
        o1 = la().la_forward_causal(q, k, v)
        o2 = la().la_forward_causal_decay(q, k, v, torch.ones(4, device="cuda"))
        torch.cuda.synchronize()
        assert la().la_get_device_status() == 0
        diff = (o1.float() - o2.float()).abs().max().item()
        assert diff <= (0.0 if d == 64 else 1.6e-2), (d, diff)


def test_causal_decay_differs_from_undecayed(orc):
    """With g < 1 the output no longer matches the undecayed causal form."""
    q, k, v = workloads.random_inputs(8555, 1, 2, 512, 64, 64, "f32")
    gamma = np.array([0.9, 0.99], dtype=np.float32)
    got = run_decay(q, k, v, gamma, "f32", 128)
    plain = orc.causal_recurrent(q, k, v)
    assert errors(got, plain)["normwise"] > 1e-2


def test_causal_decay_bf16_workload(orc):
    """The headline causal shape (B=4 H=8 N=2048 d=64, chunk 128, bf16) with
    per-head decays from 0.9 to 0.999."""
    w = workloads.CAUSAL_BF16
    q, k, v = workloads.forward_inputs(w)
    gamma = workloads.decay_gammas(w.H)
    got = run_decay(q, k, v, gamma, w.dtype, w.chunk, w.eps)
    ref = orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64), w.eps)
    e = assert_parity(got, ref, "bf16", w.name + " decay")
    print(w.name, "decay", e)


def oracle_state(orc, k, v, gamma, dk, dv):
    """Decayed state after all N tokens: the oracle's decode step from a zero state."""
    B, H, N = k.shape[:3]
    S = np.zeros((B, H, dk, dv))
    z = np.zeros((B, H, dk))
    q0 = np.zeros_like(k[:, :, 0])
    for t in range(N):
        orc.decode_step_decay(S, z, q0, k[:, :, t], v[:, :, t], gamma)
    return S, z


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,dk,dv", [(0, 64, 64), (1, 32, 32), (130, 64, 128), (700, 128, 64)])
def test_prefill_state_decay(orc, dtype, N, dk, dv):
    B, H = 2, 3
    q, k, v = workloads.random_inputs(9100 + N + dk, B, H, max(N, 1), dk, dv, dtype)
    k, v = k[:, :, :N], v[:, :, :N]
    gamma = workloads.decay_gammas(H)
    g = torch.from_numpy(gamma).cuda()
    S = torch.full((B, H, dk, dv), 7.0, device="cuda")
    z = torch.full((B, H, dk), 7.0, device="cuda")
    la().la_prefill_state_decay(to_dev(k, dtype), to_dev(v, dtype), g, S, z)
    torch.cuda.synchronize()
    if N == 0:   # overwritten with zeros
        assert not S.any() and not z.any()
        return
    Sr, zr = oracle_state(orc, k, v, gamma.astype(np.float64), dk, dv)
    es, ez = errors(from_dev(S), Sr), errors(from_dev(z), zr)
    assert es["normwise"] < 1e-5 and ez["normwise"] < 1e-5, (es, ez)


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 128, 64), (2, 3, 130, 128), (2, 3, 700, 64), (1, 4, 2000, 128),
                                     (3, 5, 1025, 64)])
def test_prefill_state_decay_tensor_core(orc, B, H, N, d):
    """bf16, dk = dv in {64, 128}, N >= 128: the tensor-core state mode with
    phi(k) times its weight in fp32, split into bf16 high and low parts."""
    q, k, v = workloads.random_inputs(9300 + N + d, B, H, N, d, d, "bf16")
    gamma = workloads.decay_gammas(H)
    g = torch.from_numpy(gamma).cuda()
    S, z = la().la_prefill_state_decay(to_dev(k, "bf16"), to_dev(v, "bf16"), g)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    Sr, zr = oracle_state(orc, k, v, gamma.astype(np.float64), d, d)
    es, ez = errors(from_dev(S), Sr), errors(from_dev(z), zr)
    assert es["normwise"] < 1e-5 and ez["normwise"] < 1e-5, (es, ez)


def test_decode_decay_after_tensor_core_prefill(orc):
    """Tensor-core decayed prefill of 300 tokens (d = 128), then 16 decayed steps."""
    B, H, P, T, d = 2, 4, 300, 16, 128
    q, k, v = workloads.random_inputs(9700, B, H, P + T, d, d, "bf16")
    gamma = np.array([0.0, 0.5, 0.99, 1.0], dtype=np.float32)
    g = torch.from_numpy(gamma).cuda()
    S, z = la().la_prefill_state_decay(to_dev(k[:, :, :P], "bf16"), to_dev(v[:, :, :P], "bf16"), g)
    full = orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64))
    for t in range(P, P + T):
        o = la().la_decode_step_decay(S, z, to_dev(q[:, :, t], "bf16"), to_dev(k[:, :, t], "bf16"),
                                      to_dev(v[:, :, t], "bf16"), g)
        torch.cuda.synchronize()
        assert_parity(from_dev(o), full[:, :, t], "bf16", ("step", t))
    Sr, zr = oracle_state(orc, k, v, gamma.astype(np.float64), d, d)
    assert errors(from_dev(S), Sr)["normwise"] < 1e-5
    assert errors(from_dev(z), zr)["normwise"] < 1e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
def test_decode_decay_continues_prefill(orc, dtype, dk, dv):
    """Decayed prefill of 40 tokens, then 24 decayed steps: every step's o equals
    the oracle's decayed causal output at that position."""
    B, H, P, T = 3, 5, 40, 24
    q, k, v = workloads.random_inputs(9500 + dk + dv, B, H, P + T, dk, dv, dtype)
    gamma = workloads.decay_gammas(H)
    g = torch.from_numpy(gamma).cuda()
    S, z = la().la_prefill_state_decay(to_dev(k[:, :, :P], dtype), to_dev(v[:, :, :P], dtype), g)
    full = orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64))
    for t in range(P, P + T):
        o = la().la_decode_step_decay(S, z, to_dev(q[:, :, t], dtype), to_dev(k[:, :, t], dtype),
                                      to_dev(v[:, :, t], dtype), g)
        torch.cuda.synchronize()
        assert_parity(from_dev(o), full[:, :, t], dtype, ("step", t))
    assert la().la_get_device_status() == 0
    Sr, zr = oracle_state(orc, k, v, gamma.astype(np.float64), dk, dv)
    assert errors(from_dev(S), Sr)["normwise"] < 1e-5
    assert errors(from_dev(z), zr)["normwise"] < 1e-5


def test_decode_decay_gamma_one_matches_undecayed():
    """g = 1 in the decayed step gives the undecayed step (1 * s is exact; only the
    compiler's choice of fused multiply-adds may differ, by an ulp)."""
    B, H, d = 4, 6, 64
    gen = torch.Generator(device="cuda").manual_seed(11)
    S0 = torch.rand((B, H, d, d), device="cuda", generator=gen)
    z0 = torch.rand((B, H, d), device="cuda", generator=gen) + 1.0
    q, k, v = (torch.randn((B, H, d), device="cuda", generator=gen).to(torch.bfloat16) for _ in range(3))
    S1, z1, S2, z2 = S0.clone(), z0.clone(), S0.clone(), z0.clone()
    o1 = la().la_decode_step(S1, z1, q, k, v)
    o2 = la().la_decode_step_decay(S2, z2, q, k, v, torch.ones(H, device="cuda"))
    torch.cuda.synchronize()
    torch.testing.assert_close(S2, S1, rtol=1e-6, atol=0)
    torch.testing.assert_close(z2, z1, rtol=1e-6, atol=0)
    torch.testing.assert_close(o2.float(), o1.float(), rtol=8e-3, atol=0)


def test_decay_output_guard_canaries():
    """Outputs of the decayed forward and step written into a sentinel-filled
    buffer: the padding on both sides stays untouched."""
    B, H, N, d, pad = 2, 3, 150, 64, 256
    gen = torch.Generator(device="cuda").manual_seed(6)
    g = torch.tensor([0.9, 0.5, 1.0], device="cuda")
    q = torch.randn((B, H, N, d), device="cuda", generator=gen).to(torch.bfloat16)
    buf = torch.full((B * H * N * d + 2 * pad,), 12345.0, dtype=torch.bfloat16, device="cuda")
    o = buf[pad:pad + B * H * N * d].view(q.shape)
    la().la_forward_causal_decay(q, q, q, g, o, chunk=64)
    qd = q[:, :, 0].contiguous()
    S = torch.zeros((B, H, d, d), device="cuda")
    z = torch.zeros((B, H, d), device="cuda")
    buf2 = torch.full((B * H * d + 2 * pad,), 12345.0, dtype=torch.bfloat16, device="cuda")
    o2 = buf2[pad:pad + B * H * d].view(qd.shape)
    la().la_decode_step_decay(S, z, qd, qd, qd, g, o2)
    torch.cuda.synchronize()
    for b, n in ((buf, B * H * N * d), (buf2, B * H * d)):
        assert torch.all(b[:pad] == 12345.0) and torch.all(b[pad + n:] == 12345.0)
    assert torch.all(torch.isfinite(o.float())) and torch.all(torch.isfinite(o2.float()))
