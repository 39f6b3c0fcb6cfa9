"""Backward pass of the causal form on the GPU vs the float64 oracle (the oracle's
gradients are pinned to finite differences of its forward).  Each gradient's max
error is scaled by the largest reference gradient of the three (dq is exactly 0
where the output cannot depend on q, e.g. N = 1): <= 1e-5 for fp32; <= 1e-2 for
bf16 inputs (exact) with fp32 arithmetic and bf16 outputs (the outputs' own
rounding, 2^-9 relative, plus fp32 accumulation)."""
import numpy as np
import pytest

import workloads
from gpu_util import from_dev, to_dev

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


TOL = {"f32": 1e-5, "bf16": 1e-2}


def check_grads(got, ref, tol, what):
    scale = max(float(np.max(np.abs(r))) for r in ref)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        d = np.abs(g - r)
        assert np.all(np.isfinite(g)), (name, what)
        assert d.max() <= tol * scale, (name, what, float(d.max()), scale)


def run_backward(q, k, v, dout, dtype, eps=1e-6):
    gq, gk, gv = la().la_backward_causal(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), to_dev(dout, dtype),
                                         eps=eps)
    torch.cuda.synchronize()
    return from_dev(gq), from_dev(gk), from_dev(gv)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,N,dk,dv", [
    (1, 1, 1, 32, 32), (2, 3, 63, 64, 64), (2, 3, 64, 64, 64), (1, 2, 65, 64, 64), (2, 2, 130, 128, 128),
    (1, 3, 300, 64, 128), (2, 2, 257, 128, 64), (1, 2, 1000, 32, 64), (2, 4, 2048, 64, 64),
    (4, 8, 2048, 64, 64),  # the benchmark's backward workload
    # bf16 d = 64 from 128 tokens runs on the tensor cores: one chunk, ragged tails
    (1, 2, 128, 64, 64), (2, 3, 200, 64, 64), (1, 2, 255, 64, 64), (2, 2, 1000, 64, 64), (1, 1, 1500, 64, 64),
    # and the narrower widths on the same 64-column tiles
    (2, 3, 300, 32, 32), (1, 2, 1000, 64, 32), (2, 2, 129, 32, 64), (4, 8, 2048, 32, 32),
])
def test_backward_matches_oracle(orc, dtype, B, H, N, dk, dv):
    """One and many chunks, ragged tails, dk != dv, every supported width."""
    q, k, v = workloads.random_inputs(20000 + N + dk + dv, B, H, N, dk, dv, dtype)
    dout = workloads.random_inputs(21000 + N, B, H, N, dv, dv, dtype)[2]
    got = run_backward(q, k, v, dout, dtype)
    ref = orc.causal_backward(q, k, v, dout)
    check_grads(got, ref, TOL[dtype], (B, H, N, dk, dv))


def test_backward_long_sequence_sampled(orc):
    """B=1 H=4 N=16384 d=64 bf16 (256 chunks through both scans): two heads
    checked against the oracle in full."""
    B, H, N, d = 1, 4, 16384, 64
    q, k, v = workloads.random_inputs(22000, B, H, N, d, d, "bf16", 0.5)
    dout = workloads.random_inputs(22001, B, H, N, d, d, "bf16", 0.5)[2]
    got = run_backward(q, k, v, dout, "bf16")
    ref = orc.causal_backward(q[:, :2], k[:, :2], v[:, :2], dout[:, :2])
    check_grads([g[:, :2] for g in got], ref, TOL["bf16"], "long")


def test_backward_first_output_only():
    """A loss on position 0 alone: o_0 = v_0, so dq = dk = 0 and dv = dout at 0 only."""
    B, H, N, d = 2, 3, 200, 64
    gen = torch.Generator(device="cuda").manual_seed(31)
    q, k, v = (torch.randn((B, H, N, d), device="cuda", generator=gen) for _ in range(3))
    dout = torch.zeros_like(v)
    dout[:, :, 0] = torch.randn((B, H, d), device="cuda", generator=gen)
    gq, gk, gv = la().la_backward_causal(q, k, v, dout)
    torch.cuda.synchronize()
    assert gq.abs().max().item() < 1e-6 and gk.abs().max().item() < 1e-6
    torch.testing.assert_close(gv[:, :, 0], dout[:, :, 0], rtol=1e-6, atol=1e-7)
    assert gv[:, :, 1:].abs().max().item() < 1e-6


def test_backward_against_autograd_of_forward_kernel_inputs():
    """Cross-check on the GPU with torch autograd of a plain fp64 quadratic form
    (masked phi(Q) phi(K)^T, row-normalised) on the same inputs."""
    B, H, N, d = 1, 2, 96, 32
    gen = torch.Generator(device="cuda").manual_seed(41)
    q, k, v, dout = (torch.randn((B, H, N, d), device="cuda", generator=gen) for _ in range(4))
    gq, gk, gv = la().la_backward_causal(q, k, v, dout)
    qq, kk, vv = (x.double().requires_grad_(True) for x in (q, k, v))
    phi = lambda x: torch.where(x > 0, x + 1, torch.exp(torch.clamp(x, max=0)))
    s = torch.tril(phi(qq) @ phi(kk).transpose(-1, -2))
    o = (s @ vv) / torch.clamp(s.sum(-1, keepdim=True), min=1e-6)
    (o * dout.double()).sum().backward()
    for g, r in ((gq, qq.grad), (gk, kk.grad), (gv, vv.grad)):
        err = (g.double() - r).abs().max() / r.abs().max()
        assert err.item() < 1e-5, err.item()


def test_backward_dependent_launches_on_a_created_stream(orc):
    """On a stream the caller created, the five launches overlap through programmatic
    dependent launch: each kernel lets the next start once its own dependency wait has
    returned, and dq and dk, dv load q, k, v, dO (dN, dd) and apply phi before their
    wait, while the scan before them still runs.  Back-to-back calls on such a
    stream, on two input sets, eager and replayed from a CUDA graph, match the
    float64 oracle (the benchmark's backward shape, B=4 H=8 N=2048 d=64)."""
    B, H, N, d = 4, 8, 2048, 64
    inputs, refs = [], []
    for i in range(2):
        q, k, v = workloads.random_inputs(24000 + i, B, H, N, d, d, "bf16")
        dout = workloads.random_inputs(24100 + i, B, H, N, d, d, "bf16")[2]
        inputs.append([to_dev(x, "bf16") for x in (q, k, v, dout)])
        refs.append(orc.causal_backward(q, k, v, dout))
    outs = [[torch.empty_like(x[j]) for j in range(3)] for x in inputs]

    def calls():
        for _ in range(2):
            for x, o in zip(inputs, outs):
                la().la_backward_causal(x[0], x[1], x[2], x[3], dq=o[0], dk=o[1], dv=o[2])

    def check(what):
        assert la().la_get_device_status() == 0
        for i, (o, ref) in enumerate(zip(outs, refs)):
            check_grads([from_dev(t) for t in o], ref, TOL["bf16"], (what, i))

    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):  # eager (the first call creates the stream's workspace)
        calls()
    torch.cuda.synchronize()
    check("eager")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    for rep in range(2):
        for o in outs:
            for t in o:
                t.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        check(("graph", rep))
