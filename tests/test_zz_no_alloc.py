"""la_forward_noncausal_noalloc: the non-causal forward for callers that may not
allocate device memory (a host program whose memory all belongs to its own pool
allocator, or a serving loop that bans allocation once running).

It must give the same answer as la_forward_noncausal.  Two calls in a row with
different shapes and dtypes show that the scratch the calls share is cleared
between them.  This file is named so that pytest collects it last.
"""
import ctypes

import pytest

import workloads
from gpu_util import assert_parity, from_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_kernelized_attention_gb300 import build
    build.build()
    import causal_kernelized_attention_gb300 as la
    return la.load_library()


def _call_noalloc(lib, q, k, v, o, dtype_code, eps=1e-6):
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.la_forward_noncausal_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, N,
                                            dk, dv, ctypes.c_float(eps), dtype_code, stream)


def test_noalloc_matches_noncausal_twice(lib):
    import causal_kernelized_attention_gb300 as la
    cases = [  # (dtype, code, B, H, N, dk, dv, seed)
        ("bf16", 1, 8, 12, 4096, 64, 64, 2),
        ("f32", 0, 2, 5, 1001, 128, 32, 9),
    ]
    for dtype, code, B, H, N, dk, dv, seed in cases:
        q, k, v = workloads.random_inputs(seed, B, H, N, dk, dv, dtype)
        dq, dk_, dv_ = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
        o_ref = la.la_forward_noncausal(dq, dk_, dv_)
        o = torch.full_like(o_ref, float("nan"))
        st = _call_noalloc(lib, dq, dk_, dv_, o, code)
        assert st == 0, la.la_status_string(st)
        torch.cuda.synchronize()
        assert_parity(from_dev(o), from_dev(o_ref), dtype, ("noalloc", dtype, B, H, N, dk, dv))


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 32 x 32 heads x 128 x 129 floats = 67.6 MB of scratch > 8 MiB: rejected before any work.
    B, H, N, d = 32, 32, 1, 128
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    assert _call_noalloc(lib, q, q, q, o, 1) == 2
    torch.cuda.synchronize()
    assert not o.any()
