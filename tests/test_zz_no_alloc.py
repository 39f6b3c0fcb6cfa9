"""la_forward_noncausal_noalloc: the non-causal forward for callers that may not
allocate device memory (a host program whose memory all belongs to its own pool
allocator, or a serving loop that bans allocation once running).

It must give the answer of the float64 oracle and of la_forward_noncausal.  Two
calls in a row with different shapes and dtypes show that the scratch the calls
share is cleared between them.  A fresh process whose first CUDA work is this
entry point shows that, once its first calls have loaded the library's array and
kernels onto the device, later calls leave the device's free memory unchanged.
This file is named so that pytest collects it last.
"""
import ctypes
import json
import os
import subprocess
import sys

import pytest

import workloads
from gpu_util import assert_parity, from_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def test_noalloc_matches_oracle_twice(lib, orc):
    """Small problems against the float64 oracle, two calls in a row (bf16 then
    fp32, other shapes): fp32 normwise <= 1e-5; bf16 max abs <= 2e-2, mean abs
    <= 2e-3 and normwise < 2e-2 (non-causal outputs are small averages)."""
    cases = [  # (dtype, code, B, H, N, dk, dv, seed)
        ("bf16", 1, 2, 3, 1000, 64, 64, 21),
        ("f32", 0, 2, 2, 257, 128, 32, 22),
    ]
    for rep in range(2):
        for dtype, code, B, H, N, dk, dv, seed in cases:
            q, k, v = workloads.random_inputs(seed, B, H, N, dk, dv, dtype)
            dq, dk_, dv_ = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
            o = torch.full(dv_.shape, float("nan"), dtype=dv_.dtype, device="cuda")
            assert _call_noalloc(lib, dq, dk_, dv_, o, code) == 0
            torch.cuda.synchronize()
            ref = orc.noncausal(q, k, v)
            e = assert_parity(from_dev(o), ref, dtype, ("noalloc vs oracle", rep, dtype, B, H, N, dk, dv))
            if dtype == "bf16":
                assert e["normwise"] < 2e-2, e


def test_noalloc_matches_noncausal_twice(lib):
    """At the non-causal workload size (B8 H12 N4096 d64, bf16) and a fp32 shape,
    against la_forward_noncausal, two calls in a row."""
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


# The child process: every tensor is allocated first; the entry point is the first
# CUDA work of this library in the process; after one call of each dtype and dk
# (which load the array and those kernels onto the device) the free device memory
# must not move across further calls.
_CHILD = r"""
import ctypes, json, sys
sys.path.insert(0, sys.argv[1])
import torch
import causal_kernelized_attention_gb300 as la
lib = la.load_library()
gen = torch.Generator(device="cuda").manual_seed(3)
def mk(B, H, N, dk, dv, dt):
    q = torch.randn((B, H, N, dk), device="cuda", generator=gen).to(dt)
    k = torch.randn((B, H, N, dk), device="cuda", generator=gen).to(dt)
    v = torch.randn((B, H, N, dv), device="cuda", generator=gen).to(dt)
    return q, k, v, torch.empty_like(v)
cases = [(mk(4, 6, 2048, 64, 64, torch.bfloat16), 1), (mk(2, 3, 999, 128, 32, torch.float32), 0),
         (mk(8, 12, 4096, 64, 64, torch.bfloat16), 1)]
def call(c):
    (q, k, v, o), code = c
    B, H, N, dk = q.shape
    st = lib.la_forward_noncausal_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, N, dk,
                                          v.shape[-1], ctypes.c_float(1e-6), code,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
torch.cuda.synchronize()
for c in cases:
    call(c)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
outs = []
for rep in range(2):
    for c in cases:
        call(c)
        torch.cuda.synchronize()
        outs.append(torch.cuda.mem_get_info()[0])
ok = all(bool(torch.isfinite(c[0][3].float()).all()) for c in cases)
print(json.dumps({"free0": free0, "free_after": outs, "finite": ok}))
"""


def test_noalloc_allocates_nothing_after_first_call_fresh_process(lib):
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-4000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["finite"], res
    assert all(f == res["free0"] for f in res["free_after"]), res
