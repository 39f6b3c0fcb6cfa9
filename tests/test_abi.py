"""The C ABI library loads, exports every declared symbol, and rejects bad
arguments before touching the GPU (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

import causal_kernelized_attention_gb300 as la
from causal_kernelized_attention_gb300 import build as la_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "la.h")

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    la_build.build()
    return la.load_library()


def test_library_is_in_tree(lib):
    assert os.path.dirname(la.lib_path()) == os.path.join(ROOT, "causal_kernelized_attention_gb300")
    assert os.path.exists(la.lib_path())


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) >= {"la_forward_causal", "la_forward_noncausal", "la_decode_step",
                          "la_prefill_state", "la_forward_causal_decay", "la_decode_step_decay",
                          "la_prefill_state_decay", "la_forward_causal_ex", "la_forward_noncausal_ex",
                          "la_decode_step_ex", "la_prefill_state_ex", "la_backward_causal",
                          "la_status_string", "la_last_cuda_error",
                          "la_get_device_status", "la_version"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in [(0, "LA_OK"), (1, "LA_ERR_INVALID_ARG"), (2, "LA_ERR_UNSUPPORTED"),
                       (3, "LA_ERR_MISALIGNED"), (4, "LA_ERR_CUDA"), (5, "LA_ERR_TIMEOUT")]:
        assert lib.la_status_string(code).decode() == name
    assert lib.la_status_string(99).decode() == "LA_ERR_UNKNOWN"
    assert lib.la_version() >= 100


# Fake pointers are only ever used in calls that must fail validation, so the
# library never dereferences or launches on them.
A = 0x100000        # 16-byte aligned
M = 0x100008        # 8-byte aligned only


def causal(lib, q=A, k=A + 0x100000, v=A + 0x200000, o=A + 0x300000, B=1, H=1, N=16, dk=64, dv=64,
           chunk=128, eps=1e-6, dtype=1):
    return lib.la_forward_causal(q, k, v, o, B, H, N, dk, dv, chunk, ctypes.c_float(eps), dtype, None)


def test_causal_validation(lib):
    assert causal(lib, q=None) == INVALID
    assert causal(lib, o=None) == INVALID
    assert causal(lib, B=-1) == INVALID
    assert causal(lib, N=-5) == INVALID
    assert causal(lib, eps=-1.0) == INVALID
    assert causal(lib, eps=float("nan")) == INVALID
    assert causal(lib, eps=float("inf")) == INVALID
    assert causal(lib, dtype=7) == INVALID
    assert causal(lib, q=M) == MISALIGNED
    assert causal(lib, o=M) == MISALIGNED
    assert causal(lib, chunk=96) == UNSUPPORTED
    assert causal(lib, chunk=0) == UNSUPPORTED
    assert causal(lib, dk=48) == UNSUPPORTED
    assert causal(lib, dv=256) == UNSUPPORTED
    # o overlapping q
    assert causal(lib, o=A + 64) == INVALID
    # empty problems are a no-op, even with NULL pointers
    assert causal(lib, N=0, q=None, k=None, v=None, o=None) == OK
    assert causal(lib, B=0, q=None, k=None, v=None, o=None) == OK


def test_noncausal_validation(lib):
    f = lib.la_forward_noncausal
    e = ctypes.c_float(1e-6)
    assert f(None, A, A, A + 0x300000, 1, 1, 8, 64, 64, e, 1, None) == INVALID
    assert f(A, A, A, M, 1, 1, 8, 64, 64, e, 1, None) == MISALIGNED
    assert f(A, A, A, A + 0x300000, 1, 1, 8, 40, 64, e, 1, None) == UNSUPPORTED
    assert f(None, None, None, None, 1, 1, 0, 64, 64, e, 1, None) == OK


def test_decode_validation(lib):
    f = lib.la_decode_step
    e = ctypes.c_float(1e-6)
    S, z, q, k, v, o = A, A + 0x800000, A + 0x900000, A + 0xA00000, A + 0xB00000, A + 0xC00000
    assert f(None, z, q, k, v, o, 2, 2, 64, 64, e, 1, None) == INVALID
    assert f(S, z, q, k, v, M, 2, 2, 64, 64, e, 1, None) == MISALIGNED
    assert f(S, z, q, k, v, o, 2, 2, 64, 96, e, 1, None) == UNSUPPORTED
    assert f(S, z, q, k, v, o, -2, 2, 64, 64, e, 1, None) == INVALID
    assert f(S, z, q, k, v, o, 2, 2, 64, 64, ctypes.c_float(-1.0), 1, None) == INVALID
    # z overlapping S
    assert f(S, S + 64, q, k, v, o, 2, 2, 64, 64, e, 1, None) == INVALID
    assert f(None, None, None, None, None, None, 0, 2, 64, 64, e, 1, None) == OK


def test_prefill_validation(lib):
    f = lib.la_prefill_state
    assert f(A, A, None, A + 0x800000, 1, 1, 8, 64, 64, 1, None) == INVALID
    assert f(A, A, M, A + 0x800000, 1, 1, 8, 64, 64, 1, None) == MISALIGNED
    assert f(A, A, A + 0x700000, A + 0x800000, 1, 1, 8, 24, 64, 1, None) == UNSUPPORTED
    assert f(None, None, None, None, 0, 1, 8, 64, 64, 1, None) == OK


def test_causal_decay_validation(lib):
    f = lib.la_forward_causal_decay
    e = ctypes.c_float(1e-6)
    q, k, v, o, g = A, A + 0x100000, A + 0x200000, A + 0x300000, A + 0x400000

    def call(q=q, k=k, v=v, o=o, g=g, B=1, H=2, N=16, dk=64, dv=64, chunk=128, eps=e, dtype=1):
        return f(q, k, v, o, g, B, H, N, dk, dv, chunk, eps, dtype, None)

    assert call(g=None) == INVALID
    assert call(g=g + 2) == MISALIGNED
    assert call(q=None) == INVALID
    assert call(o=M) == MISALIGNED
    assert call(chunk=32) == UNSUPPORTED
    assert call(dk=40) == UNSUPPORTED
    assert call(eps=ctypes.c_float(-1.0)) == INVALID
    # gamma inside o
    assert call(g=o + 16) == INVALID
    # empty problems are a no-op, even with NULL pointers and NULL gamma
    assert call(N=0, q=None, k=None, v=None, o=None, g=None) == OK


def test_decode_decay_validation(lib):
    f = lib.la_decode_step_decay
    e = ctypes.c_float(1e-6)
    S, z, q, k, v, o, g = (A, A + 0x800000, A + 0x900000, A + 0xA00000, A + 0xB00000, A + 0xC00000,
                           A + 0xD00000)
    assert f(S, z, q, k, v, o, None, 2, 2, 64, 64, e, 1, None) == INVALID
    assert f(S, z, q, k, v, o, g + 1, 2, 2, 64, 64, e, 1, None) == MISALIGNED
    assert f(S, z, q, k, v, o, S + 64, 2, 2, 64, 64, e, 1, None) == INVALID  # gamma inside S
    assert f(S, z, q, k, v, o, z + 4, 2, 2, 64, 64, e, 1, None) == INVALID   # gamma inside z
    assert f(S, z, q, k, v, o, o, 2, 2, 64, 64, e, 1, None) == INVALID       # gamma inside o
    assert f(None, z, q, k, v, o, g, 2, 2, 64, 64, e, 1, None) == INVALID
    assert f(S, z, q, k, v, o, g, 2, 2, 64, 96, e, 1, None) == UNSUPPORTED
    assert f(None, None, None, None, None, None, None, 0, 2, 64, 64, e, 1, None) == OK


def test_prefill_decay_validation(lib):
    f = lib.la_prefill_state_decay
    S, z, g = A + 0x700000, A + 0x800000, A + 0x900000
    assert f(A, A, None, S, z, 1, 1, 8, 64, 64, 1, None) == INVALID
    assert f(A, A, g + 2, S, z, 1, 1, 8, 64, 64, 1, None) == MISALIGNED
    assert f(A, A, S + 4, S, z, 1, 1, 8, 64, 64, 1, None) == INVALID   # gamma inside S
    assert f(A, A, g, M, z, 1, 1, 8, 64, 64, 1, None) == MISALIGNED
    assert f(A, A, g, S, z, 1, 1, 8, 24, 64, 1, None) == UNSUPPORTED
    assert f(None, None, None, None, None, 0, 1, 8, 64, 64, 1, None) == OK


def test_variant_validation(lib):
    """An unknown feature map, a non-finite shift or a normalize flag other than 0/1 is
    rejected by every _ex entry point before any work; so is a misaligned gamma."""
    V = la.Variant
    e = ctypes.c_float(1e-6)
    q, k, v, o = A, A + 0x100000, A + 0x200000, A + 0x300000
    S, z, g = A + 0x800000, A + 0x900000, A + 0xA00000
    bad = [V(7, 0.0, 1), V(-1, 0.0, 1), V(1, float("nan"), 1), V(2, float("inf"), 0), V(1, 0.0, 2)]
    for var in bad:
        r = ctypes.byref(var)
        assert lib.la_forward_causal_ex(q, k, v, o, None, r, 1, 2, 16, 64, 64, 128, e, 1, None) == INVALID
        assert lib.la_forward_noncausal_ex(q, k, v, o, r, 1, 2, 16, 64, 64, e, 1, None) == INVALID
        assert lib.la_decode_step_ex(S, z, q, k, v, o, None, r, 1, 2, 64, 64, e, 1, None) == INVALID
        assert lib.la_prefill_state_ex(k, v, None, r, S, z, 1, 2, 16, 64, 64, 1, None) == INVALID
    ok = ctypes.byref(V(1, 0.5, 0))
    assert lib.la_forward_causal_ex(q, k, v, o, g + 2, ok, 1, 2, 16, 64, 64, 128, e, 1, None) == MISALIGNED
    assert lib.la_forward_causal_ex(q, k, v, M, None, ok, 1, 2, 16, 64, 64, 128, e, 1, None) == MISALIGNED
    assert lib.la_forward_causal_ex(q, k, v, o, None, ok, 1, 2, 16, 48, 64, 128, e, 1, None) == UNSUPPORTED
    assert lib.la_decode_step_ex(S, z, q, k, v, o, g + 1, ok, 1, 2, 64, 64, e, 1, None) == MISALIGNED
    assert lib.la_prefill_state_ex(k, v, g + 2, ok, S, z, 1, 2, 16, 64, 64, 1, None) == MISALIGNED
    # empty problems are a no-op with any valid variant
    assert lib.la_forward_causal_ex(None, None, None, None, None, ok, 1, 2, 0, 64, 64, 128, e, 1, None) == OK
    assert lib.la_forward_noncausal_ex(None, None, None, None, ok, 0, 2, 16, 64, 64, e, 1, None) == OK


def test_backward_validation(lib):
    f = lib.la_backward_causal
    e = ctypes.c_float(1e-6)
    q, k, v, do, dq, dk, dv = (A + i * 0x100000 for i in range(7))

    def call(q=q, k=k, v=v, do=do, dq=dq, dk=dk, dv=dv, B=1, H=2, N=16, d_k=64, d_v=64, eps=e, dtype=1):
        return f(q, k, v, do, dq, dk, dv, B, H, N, d_k, d_v, eps, dtype, None)

    assert call(do=None) == INVALID
    assert call(dq=None) == INVALID
    assert call(dk=M) == MISALIGNED
    assert call(d_k=48) == UNSUPPORTED
    assert call(B=-1) == INVALID
    assert call(eps=ctypes.c_float(float("nan"))) == INVALID
    assert call(dq=k + 64) == INVALID      # an output over an input
    assert call(dv=dq) == INVALID          # two outputs on one buffer
    assert call(N=0, q=None, k=None, v=None, do=None, dq=None, dk=None, dv=None) == OK


def test_favor_validation(lib):
    e = ctypes.c_float(1e-6)
    x, w, phi = A, A + 0x100000, A + 0x200000
    ff = lib.la_favor_features
    assert ff(None, w, phi, 1, 2, 16, 64, 64, 1, None) == INVALID
    assert ff(x, None, phi, 1, 2, 16, 64, 64, 1, None) == INVALID
    assert ff(x, w, M, 1, 2, 16, 64, 64, 1, None) == MISALIGNED
    assert ff(x, w, phi, 1, 2, 16, 48, 64, 1, None) == UNSUPPORTED
    assert ff(x, w, phi, 1, 2, 16, 64, 256, 1, None) == UNSUPPORTED
    assert ff(x, w, phi, 1, 2, 16, 64, -1, 1, None) == INVALID
    assert ff(x, w, phi, 1, 2, 16, 64, 64, 5, None) == INVALID
    assert ff(x, w, x + 64, 1, 2, 16, 64, 64, 1, None) == INVALID    # phi over x
    assert ff(x, w, w - 64, 1, 2, 16, 64, 64, 1, None) == INVALID    # phi over w
    assert ff(None, None, None, 1, 2, 0, 64, 64, 1, None) == OK     # empty
    assert ff(None, None, None, 1, 2, 16, 64, 0, 1, None) == OK     # no features
    q, k, v, o, w = (A + i * 0x100000 for i in range(5))
    fc, fn = lib.la_forward_causal_favor, lib.la_forward_noncausal_favor
    assert fc(q, k, v, o, None, 1, 2, 16, 64, 64, 64, 128, e, 1, None) == INVALID
    assert fc(q, k, v, o, M, 1, 2, 16, 64, 64, 64, 128, e, 1, None) == MISALIGNED
    assert fc(q, k, v, o, w, 1, 2, 16, 64, 64, 48, 128, e, 1, None) == UNSUPPORTED
    assert fc(q, k, v, o, w, 1, 2, 16, 64, 64, 0, 128, e, 1, None) == UNSUPPORTED
    assert fc(q, k, v, o, w, 1, 2, 16, 64, 64, -2, 128, e, 1, None) == INVALID
    assert fc(q, k, v, o, w, 1, 2, 16, 64, 64, 64, 96, e, 1, None) == UNSUPPORTED
    assert fc(q, k, v, o, o + 64, 1, 2, 16, 64, 64, 64, 128, e, 1, None) == INVALID   # w over o
    assert fc(q, k, v, o, w, 1, 2, 16, 64, 64, 64, 128, ctypes.c_float(-1.0), 1, None) == INVALID
    assert fc(None, None, None, None, None, 1, 2, 0, 64, 64, 64, 128, e, 1, None) == OK
    assert fn(q, k, v, o, None, 1, 2, 16, 64, 64, 64, e, 1, None) == INVALID
    # bf16 with d = m = 64 takes the in-kernel features path: the same checks first
    assert fn(q, k, v, o, M, 1, 2, 16, 64, 64, 64, e, 1, None) == MISALIGNED
    assert fn(q, k, v, o, o + 64, 1, 2, 16, 64, 64, 64, e, 1, None) == INVALID     # w over o
    assert fn(q, k, v, o, w, 1, 2, 16, 64, 64, 64, ctypes.c_float(-1.0), 1, None) == INVALID
    assert fn(q, k, v, o, w, 1, 2, 16, 64, 32, 256, e, 1, None) == UNSUPPORTED
    assert fn(q, k, v, q + 64, w, 1, 2, 16, 64, 64, 64, e, 1, None) == INVALID      # o over q
    assert fn(None, None, None, None, None, 0, 2, 16, 64, 64, 64, e, 1, None) == OK
    fp, fd = lib.la_prefill_state_favor, lib.la_decode_step_favor
    S, z = A + 0x500000, A + 0x600000
    assert fp(k, v, None, S, z, 1, 2, 16, 64, 64, 64, 1, None) == INVALID
    assert fp(k, v, M, S, z, 1, 2, 16, 64, 64, 64, 1, None) == MISALIGNED
    assert fp(k, v, w, S, z, 1, 2, 16, 64, 64, 48, 1, None) == UNSUPPORTED
    assert fp(k, v, w, S, z, 1, 2, 16, 0, 64, 64, 1, None) == UNSUPPORTED
    assert fp(k, v, S + 64, S, z, 1, 2, 16, 64, 64, 64, 1, None) == INVALID        # w over S
    assert fp(k, v, w, S, z, 1, 2, 16, 64, 64, 64, 7, None) == INVALID
    assert fp(None, None, None, S, z, 0, 2, 16, 64, 64, 64, 1, None) == OK         # empty
    assert fd(S, z, q, k, v, o, None, 1, 2, 64, 64, 64, e, 1, None) == INVALID
    assert fd(S, z, q, k, v, o, M, 1, 2, 64, 64, 64, e, 1, None) == MISALIGNED
    assert fd(S, z, q, k, v, o, w, 1, 2, 64, 64, 256, e, 1, None) == UNSUPPORTED
    assert fd(S, z, q, k, v, o, o + 64, 1, 2, 64, 64, 64, e, 1, None) == INVALID   # w over o
    assert fd(S, z, q, k, v, q + 64, w, 1, 2, 64, 64, 64, e, 1, None) == INVALID   # o over q
    assert fd(S, z, q, k, v, o, w, 1, 2, 64, 64, 64, ctypes.c_float(float("nan")), 1, None) == INVALID
    assert fd(None, None, None, None, None, None, None, 1, 0, 64, 64, 64, e, 1, None) == OK


def test_binding_raises_without_cuda_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 64)
    with pytest.raises(ValueError):
        la.la_forward_causal(q, q, q, q.clone())
