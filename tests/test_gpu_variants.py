"""Feature-map and normaliser variants on the GPU vs the float64 oracle.

Maps: elu + 1, max(x, 0) + c ("Linear attention", What the pieces are for: ReLU;
"26. Linear (Kernelized) Attention", Key Functions & Tricks: relu(x) + eps) and
x + c ("Linear Attention -- Math + Variants", Feature-map families: identity-plus-
shift); with or without the phi(q)^T z normaliser (same page, Implementation
reality); with or without the per-head decay.  Every call goes through the C ABI.

Tolerances: normalised outputs are weighted averages of v, so the usual bounds
hold (fp32 normwise 1e-5; bf16 max abs 2e-2, mean abs 2e-3).  Without the
normaliser |o| grows with the number of keys, so those outputs are held to a
normwise bound: max|gpu - oracle| / max|oracle| <= 1e-5 (fp32), <= 2e-2 (bf16).
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


# (map, shift, normalize): identity maps are only meaningful without the normaliser
# (phi(q).phi(k) can be negative), as in retention-style layers.
VARIANTS = [("relu", 0.0, True), ("relu", 0.25, True), ("relu", 0.0, False), ("identity", 0.5, False),
            ("elu1", 0.0, False)]


def check(got, ref, dtype, normalize, what):
    if normalize:
        return assert_parity(got, ref, dtype, what)
    e = errors(got, ref)
    assert e["finite"], what
    assert e["normwise"] <= (1e-5 if dtype == "f32" else 2e-2), (what, e)
    return e


def gamma_dev(gamma):
    return None if gamma is None else torch.from_numpy(np.asarray(gamma, dtype=np.float32)).cuda()


@pytest.mark.parametrize("fmap,shift,normalize", VARIANTS)
@pytest.mark.parametrize("dtype,B,H,N,d,chunk", [
    ("bf16", 2, 3, 300, 64, 128), ("bf16", 1, 4, 1000, 128, 128), ("bf16", 2, 3, 2000, 64, 128),
    ("bf16", 1, 2, 20000, 64, 128), ("bf16", 2, 3, 257, 64, 64), ("f32", 2, 3, 300, 64, 128),
    ("f32", 1, 2, 129, 32, 64),
])
def test_causal_variant(orc, fmap, shift, normalize, dtype, B, H, N, d, chunk):
    """Tensor-core shapes (bf16, chunk 128: short and scan modes) and CUDA-core shapes."""
    q, k, v = workloads.random_inputs(15000 + N + d + chunk, B, H, N, d, d, dtype)
    o = la().la_forward_causal_ex(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), feature_map=fmap,
                                  shift=shift, normalize=normalize, chunk=chunk)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.causal_general(q, k, v, fmap=fmap, shift=shift, normalize=normalize)
    check(from_dev(o), ref, dtype, normalize, (fmap, shift, normalize, N, d))


@pytest.mark.parametrize("fmap,shift,normalize", [("identity", 0.0, False), ("relu", 0.1, True),
                                                  ("relu", 0.0, False)])
@pytest.mark.parametrize("B,H,N,d", [(2, 4, 1000, 64), (1, 4, 3000, 128), (1, 4, 20000, 64)])
def test_causal_decay_variant(orc, fmap, shift, normalize, B, H, N, d):
    """Decay with the other maps on the tensor-core path; identity without the
    normaliser is the retention form (a fixed per-head decay, no feature map)."""
    q, k, v = workloads.random_inputs(16000 + N + d, B, H, N, d, d, "bf16")
    gamma = workloads.decay_gammas(H)
    o = la().la_forward_causal_ex(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"), gamma=gamma_dev(gamma),
                                  feature_map=fmap, shift=shift, normalize=normalize)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.causal_general(q, k, v, gamma=gamma.astype(np.float64), fmap=fmap, shift=shift, normalize=normalize)
    check(from_dev(o), ref, "bf16", normalize, (fmap, normalize, N, d))


def test_causal_relu_dead_queries_give_zero():
    """ReLU without shift: queries with no positive component give o = 0 exactly."""
    B, H, N, d = 1, 2, 300, 64
    gen = torch.Generator(device="cuda").manual_seed(17)
    q = -(torch.rand((B, H, N, d), device="cuda", generator=gen)).to(torch.bfloat16)
    k, v = (torch.randn((B, H, N, d), device="cuda", generator=gen).to(torch.bfloat16) for _ in range(2))
    for normalize in (True, False):
        o = la().la_forward_causal_ex(q, k, v, feature_map="relu", shift=0.0, normalize=normalize)
        torch.cuda.synchronize()
        assert torch.all(o == 0)


@pytest.mark.parametrize("fmap,shift,normalize", VARIANTS)
@pytest.mark.parametrize("dtype,B,H,N,d", [("bf16", 2, 6, 4096, 64), ("bf16", 2, 3, 1000, 128),
                                           ("f32", 2, 3, 500, 64)])
def test_noncausal_variant(orc, fmap, shift, normalize, dtype, B, H, N, d):
    q, k, v = workloads.random_inputs(17000 + N + d, B, H, N, d, d, dtype)
    o = la().la_forward_noncausal_ex(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), feature_map=fmap,
                                     shift=shift, normalize=normalize)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    ref = orc.noncausal_general(q, k, v, fmap=fmap, shift=shift, normalize=normalize)
    e = check(from_dev(o), ref, dtype, normalize, (fmap, normalize, N, d))
    if normalize and dtype == "bf16":  # non-causal outputs are small averages: also normwise
        assert e["normwise"] < 2e-2, e


@pytest.mark.parametrize("fmap,shift", [("relu", 0.0), ("relu", 0.3), ("identity", 0.2)])
@pytest.mark.parametrize("dtype,B,H,N,d", [("bf16", 2, 3, 700, 64), ("bf16", 1, 4, 2000, 128),
                                           ("f32", 2, 3, 300, 64), ("bf16", 2, 3, 50, 32)])
@pytest.mark.parametrize("decay", [False, True])
def test_prefill_state_variant(orc, fmap, shift, dtype, B, H, N, d, decay):
    q, k, v = workloads.random_inputs(18000 + N + d, B, H, N, d, d, dtype)
    gamma = workloads.decay_gammas(H) if decay else None
    S, z = la().la_prefill_state_ex(to_dev(k, dtype), to_dev(v, dtype), gamma=gamma_dev(gamma),
                                    feature_map=fmap, shift=shift)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    Sr, zr = orc.prefill_state_general(k, v, gamma=None if gamma is None else gamma.astype(np.float64),
                                       fmap=fmap, shift=shift)
    es, ez = errors(from_dev(S), Sr), errors(from_dev(z), zr)
    assert es["normwise"] < 1e-5 and ez["normwise"] < 1e-5, (es, ez)


@pytest.mark.parametrize("fmap,shift,normalize", [("relu", 0.1, True), ("identity", 0.0, False),
                                                  ("relu", 0.0, False)])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("bf16", 32)])
def test_decode_variant_continues_prefill(orc, fmap, shift, normalize, dtype, d):
    """Variant prefill (tensor cores where the shape allows), then 12 variant steps with
    a per-head decay: every step equals the oracle's general causal form there."""
    B, H, P, T = 2, 4, 200, 12
    q, k, v = workloads.random_inputs(19000 + d, B, H, P + T, d, d, dtype)
    gamma = np.array([0.9, 0.5, 1.0, 0.99], dtype=np.float32)
    g = gamma_dev(gamma)
    S, z = la().la_prefill_state_ex(to_dev(k[:, :, :P], dtype), to_dev(v[:, :, :P], dtype), gamma=g,
                                    feature_map=fmap, shift=shift)
    full = orc.causal_general(q, k, v, gamma=gamma.astype(np.float64), fmap=fmap, shift=shift, normalize=normalize)
    for t in range(P, P + T):
        o = la().la_decode_step_ex(S, z, to_dev(q[:, :, t], dtype), to_dev(k[:, :, t], dtype),
                                   to_dev(v[:, :, t], dtype), gamma=g, feature_map=fmap, shift=shift,
                                   normalize=normalize)
        torch.cuda.synchronize()
        check(from_dev(o), full[:, :, t], dtype, normalize, (fmap, t))
    assert la().la_get_device_status() == 0


def test_default_variant_is_the_plain_kernel():
    """la_*_ex with the default variant and no decay returns what the plain entry
    points return, bit for bit (the same kernels run)."""
    gen = torch.Generator(device="cuda").manual_seed(23)
    q, k, v = ((torch.randn((2, 4, 1500, 64), device="cuda", generator=gen) * 0.5).to(torch.bfloat16)
               for _ in range(3))
    assert torch.equal(la().la_forward_causal(q, k, v), la().la_forward_causal_ex(q, k, v))
    assert torch.equal(la().la_forward_noncausal(q, k, v), la().la_forward_noncausal_ex(q, k, v))
    S1, z1 = la().la_prefill_state(k, v)
    S2, z2 = la().la_prefill_state_ex(k, v)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2) and torch.equal(z1, z2)
