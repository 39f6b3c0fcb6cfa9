"""Feature widths other than dk = dv in {64, 128} on the tensor cores (needs a GB300).

The signature of "26. Linear (Kernelized) Attention" takes q, k [.., dk] and
v [.., dv] with dk != dv; the library accepts dk, dv in {32, 64, 128}.  For
bf16 with N >= 128 the widths other than dk = dv in {64, 128} run on the tensor-core
kernels on tiles of the next width (64 or 128): TMA fills the columns past each
width with zeros and clips them from the stores, and the kernels zero phi(K)'s
extra columns (phi(0) is 1 for elu + 1).  Every call goes through the C ABI and
is compared with the float64 oracle at the bf16 tolerances (max abs 2e-2, mean
abs 2e-3; normwise 2e-2 where the normaliser is off).  A profiler pass checks
that the tensor-core kernels, not the CUDA-core ones, ran.
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


def kernels_of(fn):
    """Names of the CUDA kernels fn launches (empty if the profiler records none;
    its first session in a process can come back empty, so an empty one is retried)."""
    from torch.profiler import ProfilerActivity, profile
    for _ in range(2):
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
        if names:
            return names
    return []


def check(got, ref, normalize, what):
    if normalize:
        return assert_parity(got, ref, "bf16", what)
    e = errors(got, ref)
    assert e["finite"], what
    assert e["normwise"] <= 2e-2, (what, e)
    return e


@pytest.mark.parametrize("B,H,N,dk,dv", [
    (2, 3, 129, 32, 32), (1, 2, 1000, 32, 32), (4, 8, 2048, 32, 32), (2, 2, 300, 64, 128),
    (1, 3, 2000, 128, 64), (1, 2, 5000, 32, 128), (2, 1, 700, 128, 32), (1, 1, 20000, 64, 32),
    (3, 2, 128, 32, 64),
])
def test_causal_widths(orc, B, H, N, dk, dv):
    """Short mode (segments summing their own prefix) and scan mode (chained
    segments), ragged tails, one-chunk heads; tiles of 64 and of 128 columns."""
    q, k, v = workloads.random_inputs(30000 + N + dk + 3 * dv, B, H, N, dk, dv, "bf16")
    o = la().la_forward_causal(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), chunk=128)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    e = assert_parity(from_dev(o), orc.causal_recurrent(q, k, v), "bf16", (B, H, N, dk, dv))
    assert e["normwise"] < 2e-2, e


@pytest.mark.parametrize("fmap,shift,normalize", [("relu", 0.25, True), ("identity", 0.5, False),
                                                  ("elu1", 0.0, False), ("relu", 0.0, True)])
@pytest.mark.parametrize("B,H,N,dk,dv", [(2, 3, 1000, 32, 32), (1, 2, 3000, 64, 128), (2, 2, 400, 128, 32)])
def test_causal_widths_variants(orc, fmap, shift, normalize, B, H, N, dk, dv):
    """Maps whose phi(0) is not 0 (a shift, elu + 1) are where the extra columns of
    phi(K) must be zeroed; without the normaliser nothing hides a phantom feature."""
    q, k, v = workloads.random_inputs(31000 + N + dk + dv, B, H, N, dk, dv, "bf16")
    o = la().la_forward_causal_ex(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), feature_map=fmap,
                                  shift=shift, normalize=normalize)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.causal_general(q, k, v, fmap=fmap, shift=shift, normalize=normalize)
    check(from_dev(o), ref, normalize, (fmap, shift, normalize, N, dk, dv))


@pytest.mark.parametrize("fmap,shift,normalize", [("elu1", 0.0, True), ("relu", 0.1, True),
                                                  ("identity", 0.0, False)])
@pytest.mark.parametrize("B,H,N,dk,dv", [(2, 4, 1000, 32, 64), (1, 4, 3000, 128, 64), (1, 2, 9000, 32, 32)])
def test_causal_widths_decay(orc, fmap, shift, normalize, B, H, N, dk, dv):
    q, k, v = workloads.random_inputs(32000 + N + dk + dv, B, H, N, dk, dv, "bf16")
    gamma = workloads.decay_gammas(H)
    o = la().la_forward_causal_ex(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"),
                                  gamma=torch.from_numpy(gamma.astype(np.float32)).cuda(), feature_map=fmap,
                                  shift=shift, normalize=normalize)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.causal_general(q, k, v, gamma=gamma.astype(np.float64), fmap=fmap, shift=shift, normalize=normalize)
    check(from_dev(o), ref, normalize, ("decay", fmap, N, dk, dv))


@pytest.mark.parametrize("B,H,N,dk,dv", [
    (2, 3, 1000, 32, 32), (4, 40, 4173, 32, 32), (2, 2, 300, 64, 128), (1, 3, 2000, 128, 64),
    (1, 2, 65536, 32, 128), (64, 16, 128, 32, 64),
])
def test_noncausal_widths(orc, B, H, N, dk, dv):
    """One and many key splits per head, many one-chunk heads."""
    q, k, v = workloads.random_inputs(33000 + N + dk + dv, B, H, N, dk, dv, "bf16")
    o = la().la_forward_noncausal(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"))
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    e = assert_parity(from_dev(o), orc.noncausal(q, k, v), "bf16", (B, H, N, dk, dv))
    assert e["normwise"] < 2e-2, e


@pytest.mark.parametrize("fmap,shift,normalize", [("relu", 0.25, True), ("identity", 0.5, False)])
def test_noncausal_widths_variants(orc, fmap, shift, normalize):
    B, H, N, dk, dv = 2, 3, 1500, 32, 64
    q, k, v = workloads.random_inputs(34000 + N, B, H, N, dk, dv, "bf16")
    o = la().la_forward_noncausal_ex(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), feature_map=fmap,
                                     shift=shift, normalize=normalize)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.noncausal_general(q, k, v, fmap=fmap, shift=shift, normalize=normalize)
    check(from_dev(o), ref, normalize, (fmap, shift, normalize))


@pytest.mark.parametrize("path,dk,dv", [("causal", 32, 32), ("causal", 64, 128), ("noncausal", 32, 64),
                                        ("noncausal", 128, 64)])
def test_widths_run_on_the_tensor_cores(path, dk, dv):
    B, H, N = 2, 3, 1000
    gen = torch.Generator(device="cuda").manual_seed(dk + dv)
    q, k = (torch.randn((B, H, N, dk), device="cuda", generator=gen).to(torch.bfloat16) for _ in range(2))
    v = torch.randn((B, H, N, dv), device="cuda", generator=gen).to(torch.bfloat16)
    call = (lambda: la().la_forward_causal(q, k, v, chunk=128)) if path == "causal" else \
        (lambda: la().la_forward_noncausal(q, k, v))
    call()
    torch.cuda.synchronize()
    names = kernels_of(call)
    if not names:
        pytest.skip("the profiler recorded no kernels")
    want = "causal_tc_kernel" if path == "causal" else "noncausal_tc_kernel"
    assert any(want in n for n in names), names
    assert not any("simt" in n for n in names), names


@pytest.mark.parametrize("B,H,N,dk,dv", [
    (2, 3, 700, 32, 32), (1, 4, 2000, 64, 128), (2, 2, 300, 128, 32), (16, 20, 130, 32, 64),
    (1, 2, 65536, 32, 128),
])
@pytest.mark.parametrize("fmap,shift,decay", [("elu1", 0.0, False), ("elu1", 0.0, True), ("relu", 0.3, False)])
def test_prefill_state_widths(orc, B, H, N, dk, dv, fmap, shift, decay):
    """The prefix state [dk, dv] and z [dk] from the D-wide sums: one key split per
    head (written by the split itself: 16 x 20 heads of one chunk) and many (summed
    by the CTA that completes the last); the state rows past dk, fed by phi(0), are
    not written."""
    _, k, v = workloads.random_inputs(35000 + N + dk + dv, B, H, N, dk, dv, "bf16")
    gamma = workloads.decay_gammas(H) if decay else None
    S, z = la().la_prefill_state_ex(to_dev(k, "bf16"), to_dev(v, "bf16"),
                                    gamma=None if gamma is None else torch.from_numpy(gamma).cuda(),
                                    feature_map=fmap, shift=shift)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    assert S.shape == (B, H, dk, dv) and z.shape == (B, H, dk)
    Sr, zr = orc.prefill_state_general(k, v, gamma=None if gamma is None else gamma.astype(np.float64),
                                       fmap=fmap, shift=shift)
    es, ez = errors(from_dev(S), Sr), errors(from_dev(z), zr)
    assert es["normwise"] < 1e-5 and ez["normwise"] < 1e-5, (es, ez)


@pytest.mark.parametrize("dk,dv", [(32, 32), (32, 64), (64, 32)])
def test_backward_widths_run_on_the_tensor_cores(dk, dv):
    """The backward at widths up to 64 runs the five tensor-core launches (its parity
    against the oracle is in test_gpu_backward.py)."""
    B, H, N = 2, 3, 1000
    gen = torch.Generator(device="cuda").manual_seed(dk * dv)
    q, k = (torch.randn((B, H, N, dk), device="cuda", generator=gen).to(torch.bfloat16) for _ in range(2))
    v, do = (torch.randn((B, H, N, dv), device="cuda", generator=gen).to(torch.bfloat16) for _ in range(2))
    call = lambda: la().la_backward_causal(q, k, v, do)
    call()
    torch.cuda.synchronize()
    names = kernels_of(call)
    if not names:
        pytest.skip("the profiler recorded no kernels")
    assert sum("bwd_tc" in n for n in names) == 5, names
