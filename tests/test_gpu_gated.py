"""Gated state, one gate per key feature, on the GPU vs the float64 oracle.

S_t = Diag(alpha_t) S_{t-1} + phi(k_t) v_t^T and z gated alike ("Linear
Attention", What is actually lost; "Linear Attention -- Math + Variants", RetNet
and gated linear attention), the gate alpha an input.  Every call goes through
the C ABI.  Tolerances as for the other forms: fp32 normwise <= 1e-5; bf16 max
abs <= 2e-2 and mean abs <= 2e-3 (outputs stay convex combinations of the v_j);
the state of the prefix and of the decode steps (fp32) normwise <= 1e-5.
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


def gates(seed, shape, lo=0.8):
    """Per-(token, feature) gates in [lo, 1), float32 (exact on both sides)."""
    return np.random.default_rng(seed).uniform(lo, 1.0, size=shape).astype(np.float32)


def dev_f32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,N,dk,dv", [
    (1, 1, 1, 32, 32), (2, 3, 31, 64, 64), (2, 3, 33, 64, 64), (1, 2, 300, 128, 64), (2, 2, 257, 32, 128),
    (1, 3, 1000, 64, 32), (2, 2, 2048, 128, 128), (4, 8, 2048, 64, 64),
])
def test_gated_causal_matches_oracle(orc, dtype, B, H, N, dk, dv):
    """One and many 32-token chunks, ragged tails, dk != dv, every width, and the
    headline shape."""
    q, k, v = workloads.random_inputs(60000 + N + dk + dv, B, H, N, dk, dv, dtype)
    a = gates(60001 + N, (B, H, N, dk))
    o = la().la_forward_causal_gated(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), dev_f32(a))
    torch.cuda.synchronize()
    ref = orc.causal_gated_recurrent(q, k, v, a.astype(np.float64))
    assert_parity(from_dev(o), ref, dtype, (B, H, N, dk, dv))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gated_small_gates(orc, dtype):
    """Gates drawn from [0, 1): products over a few tokens underflow; the chunked form
    never divides by a product of gates, so it matches the recurrence."""
    B, H, N, d = 2, 3, 1000, 64
    q, k, v = workloads.random_inputs(60500, B, H, N, d, d, dtype)
    a = gates(60501, (B, H, N, d), lo=0.0)
    o = la().la_forward_causal_gated(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), dev_f32(a))
    torch.cuda.synchronize()
    assert_parity(from_dev(o), orc.causal_gated_recurrent(q, k, v, a.astype(np.float64)), dtype, "small gates")


def test_gated_special_gates(orc):
    """Gates of 1 give la_forward_causal; gates of gamma[h] give the decayed form;
    gates of 0 give o = v; closing one feature keeps the others' history."""
    B, H, N, d = 2, 3, 500, 64
    q, k, v = workloads.random_inputs(61000, B, H, N, d, d, "f32")
    qd, kd, vd = to_dev(q, "f32"), to_dev(k, "f32"), to_dev(v, "f32")
    ones = torch.ones((B, H, N, d), device="cuda")
    o1 = la().la_forward_causal_gated(qd, kd, vd, ones)
    o_plain = la().la_forward_causal(qd, kd, vd, chunk=64)
    g = workloads.decay_gammas(H)
    gam = torch.from_numpy(g).cuda()
    o2 = la().la_forward_causal_gated(qd, kd, vd, gam.view(1, H, 1, 1).expand(B, H, N, d).contiguous())
    o_dec = la().la_forward_causal_decay(qd, kd, vd, gam, chunk=64)
    o0 = la().la_forward_causal_gated(qd, kd, vd, torch.zeros_like(ones))
    a = np.ones((B, H, N, d), np.float32)
    a[..., 5] = 0.0
    o3 = la().la_forward_causal_gated(qd, kd, vd, dev_f32(a))
    torch.cuda.synchronize()
    assert errors(from_dev(o1), from_dev(o_plain))["normwise"] < 1e-5
    assert errors(from_dev(o2), from_dev(o_dec))["normwise"] < 1e-5
    assert errors(from_dev(o0), v)["normwise"] < 1e-5
    assert_parity(from_dev(o3), orc.causal_gated_recurrent(q, k, v, a.astype(np.float64)), "f32", "one feature closed")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
def test_gated_prefill_and_decode(orc, dtype, dk, dv):
    """Prefill 40 tokens, then 20 decode steps: every step's o against the oracle's
    gated recurrence over the whole sequence, the final state against its prefix state."""
    B, H, P, T = 3, 5, 40, 20
    q, k, v = workloads.random_inputs(62000 + dk + dv, B, H, P + T, dk, dv, dtype)
    a = gates(62001 + dk, (B, H, P + T, dk))
    S, z = la().la_prefill_state_gated(to_dev(k[:, :, :P], dtype), to_dev(v[:, :, :P], dtype), dev_f32(a[:, :, :P]))
    torch.cuda.synchronize()
    Sr, zr = orc.prefill_state_gated(k[:, :, :P], v[:, :, :P], a[:, :, :P].astype(np.float64))
    assert errors(from_dev(S), Sr)["normwise"] < 1e-5 and errors(from_dev(z), zr)["normwise"] < 1e-5
    full = orc.causal_gated_recurrent(q, k, v, a.astype(np.float64))
    for t in range(P, P + T):
        o = la().la_decode_step_gated(S, z, to_dev(q[:, :, t], dtype), to_dev(k[:, :, t], dtype),
                                      to_dev(v[:, :, t], dtype), dev_f32(a[:, :, t]))
        torch.cuda.synchronize()
        assert_parity(from_dev(o), full[:, :, t], dtype, ("step", t))
    Sr, zr = orc.prefill_state_gated(k, v, a.astype(np.float64))
    assert errors(from_dev(S), Sr)["normwise"] < 1e-5 and errors(from_dev(z), zr)["normwise"] < 1e-5


def test_gated_empty_prefix_and_canaries():
    """N = 0 writes a zero state; outputs inside sentinel-filled buffers leave the
    padding untouched."""
    B, H, N, d = 2, 3, 150, 64
    k0 = torch.empty((B, H, 0, d), device="cuda")
    S = torch.full((B, H, d, d), 7.0, device="cuda")
    z = torch.full((B, H, d), 7.0, device="cuda")
    la().la_prefill_state_gated(k0, k0, torch.empty((B, H, 0, d), device="cuda"), S, z)
    torch.cuda.synchronize()
    assert not S.any() and not z.any()
    pad = 256
    gen = torch.Generator(device="cuda").manual_seed(8)
    x = torch.randn((B, H, N, d), device="cuda", generator=gen).to(torch.bfloat16)
    a = torch.rand((B, H, N, d), device="cuda", generator=gen)
    buf = torch.full((B * H * N * d + 2 * pad,), 12345.0, dtype=torch.bfloat16, device="cuda")
    o = buf[pad:pad + B * H * N * d].view(B, H, N, d)
    la().la_forward_causal_gated(x, x, x, a, o=o)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345.0) and torch.all(buf[-pad:] == 12345.0)
    assert torch.all(torch.isfinite(o.float()))


def test_gated_argument_checks():
    q = torch.zeros((1, 2, 10, 64), device="cuda")
    with pytest.raises(ValueError):
        la().la_forward_causal_gated(q, q, q, torch.ones((1, 2, 10, 32), device="cuda"))
    lib = la().load_library()
    import ctypes
    o = torch.empty_like(q)
    a = torch.ones_like(q)
    st = lib.la_forward_causal_gated(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), None, 1, 2, 10, 64, 64,
                                     ctypes.c_float(1e-6), 0, None)
    assert st == 1  # a missing gate
    st = lib.la_forward_causal_gated(q.data_ptr(), q.data_ptr(), q.data_ptr(), a.data_ptr(), a.data_ptr(), 1, 2, 10,
                                     64, 64, ctypes.c_float(1e-6), 0, None)
    assert st == 1  # the output overlaps the gate
