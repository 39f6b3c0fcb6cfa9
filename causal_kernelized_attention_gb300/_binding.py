"""ctypes marshalling for liblinattn.so (argument checks and pointers only)."""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

LA_F32 = 0
LA_BF16 = 1

_STATUS_NAMES = {0: "LA_OK", 1: "LA_ERR_INVALID_ARG", 2: "LA_ERR_UNSUPPORTED", 3: "LA_ERR_MISALIGNED",
                 4: "LA_ERR_CUDA", 5: "LA_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class LAError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = "%s returned %s" % (fn, _STATUS_NAMES.get(status, status))
        if cuda_error:
            msg += " (cudaError %d)" % cuda_error
        super().__init__(msg)


class Variant(ctypes.Structure):
    """la_variant: feature map (LA_PHI_ELU1 / LA_PHI_RELU / LA_PHI_IDENTITY), its shift,
    and whether the output is divided by max(phi(q)^T z, eps)."""
    _fields_ = [("feature_map", ctypes.c_int), ("shift", ctypes.c_float), ("normalize", ctypes.c_int)]


LA_PHI_ELU1, LA_PHI_RELU, LA_PHI_IDENTITY = 0, 1, 2
_FMAPS = {"elu1": LA_PHI_ELU1, "relu": LA_PHI_RELU, "identity": LA_PHI_IDENTITY}


def _variant(feature_map, shift, normalize):
    """A la_variant by reference, or None for the default (elu + 1, normalised)."""
    fm = _FMAPS[feature_map] if isinstance(feature_map, str) else int(feature_map)
    if fm == LA_PHI_ELU1 and normalize:
        return None
    return ctypes.byref(Variant(fm, float(shift), 1 if normalize else 0))


def lib_path() -> str:
    return LIB_PATH


def _declare(lib):
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sigs = {
        "la_forward_causal": [P, P, P, P, I, I, I, I, I, I, F, I, P],
        "la_forward_noncausal": [P, P, P, P, I, I, I, I, I, F, I, P],
        "la_forward_noncausal_noalloc": [P, P, P, P, I, I, I, I, I, F, I, P],
        "la_decode_step": [P, P, P, P, P, P, I, I, I, I, F, I, P],
        "la_prefill_state": [P, P, P, P, I, I, I, I, I, I, P],
        "la_forward_causal_decay": [P, P, P, P, P, I, I, I, I, I, I, F, I, P],
        "la_decode_step_decay": [P, P, P, P, P, P, P, I, I, I, I, F, I, P],
        "la_prefill_state_decay": [P, P, P, P, P, I, I, I, I, I, I, P],
        "la_forward_causal_ex": [P, P, P, P, P, P, I, I, I, I, I, I, F, I, P],
        "la_forward_noncausal_ex": [P, P, P, P, P, I, I, I, I, I, F, I, P],
        "la_decode_step_ex": [P, P, P, P, P, P, P, P, I, I, I, I, F, I, P],
        "la_prefill_state_ex": [P, P, P, P, P, P, I, I, I, I, I, I, P],
        "la_backward_causal": [P, P, P, P, P, P, P, I, I, I, I, I, F, I, P],
        "la_favor_features": [P, P, P, I, I, I, I, I, I, P],
        "la_forward_causal_favor": [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P],
        "la_forward_noncausal_favor": [P, P, P, P, P, I, I, I, I, I, I, F, I, P],
        "la_prefill_state_favor": [P, P, P, P, P, I, I, I, I, I, I, I, P],
        "la_decode_step_favor": [P, P, P, P, P, P, P, I, I, I, I, I, F, I, P],
        "la_forward_causal_gated": [P, P, P, P, P, I, I, I, I, I, F, I, P],
        "la_prefill_state_gated": [P, P, P, P, P, I, I, I, I, I, I, P],
        "la_decode_step_gated": [P, P, P, P, P, P, P, I, I, I, I, F, I, P],
        "la_get_device_status": [P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.la_status_string.argtypes = [ctypes.c_int]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_last_cuda_error.argtypes = []
    lib.la_last_cuda_error.restype = ctypes.c_int
    lib.la_version.argtypes = []
    lib.la_version.restype = ctypes.c_int
    lib.la_kernel_launches.argtypes = []
    lib.la_kernel_launches.restype = ctypes.c_ulonglong
    lib.la_test_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.la_test_set_wait_limit_ns.restype = None
    lib.la_test_drop_publication.argtypes = [ctypes.c_longlong]
    lib.la_test_drop_publication.restype = None
    return lib


def load_library(path: str = None):
    """Load liblinattn.so (built by ``build.py`` / ``__graft_entry__.build()``).

    Raises OSError with a clear message when the library has not been built.
    """
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise OSError("liblinattn.so not found at %s: build it with "
                          "`python -m causal_kernelized_attention_gb300.build`" % p)
        lib = _declare(ctypes.CDLL(p))
        if path is None:
            _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != 0:
        raise LAError(fn, status, load_library().la_last_cuda_error() if status == 4 else 0)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError("q, k, v, o must be float32 or bfloat16, got %s" % t.dtype)


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _same_dtype(*ts):
    d = ts[0].dtype
    for t in ts[1:]:
        if t.dtype != d:
            raise TypeError("q, k, v, o must share one dtype")


def la_forward_causal(q, k, v, o=None, chunk: int = 128, eps: float = 1e-6, stream=None):
    """Causal forward; q, k [B,H,N,dk], v [B,H,N,dv]; returns o [B,H,N,dv]."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, N, dk) or tuple(v.shape[:-1]) != (B, H, N) or tuple(o.shape) != (B, H, N, dv):
        raise ValueError("shape mismatch")
    st = load_library().la_forward_causal(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                          B, H, N, dk, dv, int(chunk), float(eps), _dtype_code(q),
                                          _stream_ptr(stream))
    _check("la_forward_causal", st)
    return o


def la_forward_noncausal(q, k, v, o=None, eps: float = 1e-6, stream=None):
    """Non-causal forward; q, k [B,H,N,dk], v [B,H,N,dv]; returns o [B,H,N,dv]."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, N, dk) or tuple(v.shape[:-1]) != (B, H, N) or tuple(o.shape) != (B, H, N, dv):
        raise ValueError("shape mismatch")
    st = load_library().la_forward_noncausal(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                             B, H, N, dk, dv, float(eps), _dtype_code(q), _stream_ptr(stream))
    _check("la_forward_noncausal", st)
    return o


def la_forward_noncausal_noalloc(q, k, v, o, eps: float = 1e-6, stream=None):
    """Non-causal forward using the library's fixed scratch array (no device
    allocation by the library).  `o` must be supplied by the caller."""
    _need_cuda(q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, N, dk) or tuple(v.shape[:-1]) != (B, H, N) or tuple(o.shape) != (B, H, N, dv):
        raise ValueError("shape mismatch")
    st = load_library().la_forward_noncausal_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                     B, H, N, dk, dv, float(eps), _dtype_code(q),
                                                     _stream_ptr(stream))
    _check("la_forward_noncausal_noalloc", st)
    return o


def la_decode_step(S, z, q, k, v, o=None, eps: float = 1e-6, stream=None):
    """One decode step; S [B,H,dk,dv], z [B,H,dk] fp32 updated in place; returns o [B,H,dv]."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(S, z, q, k, v, o)
    _same_dtype(q, k, v, o)
    if S.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("S and z must be float32")
    B, H, dk = q.shape
    dv = v.shape[-1]
    if tuple(S.shape) != (B, H, dk, dv) or tuple(z.shape) != (B, H, dk) or tuple(k.shape) != (B, H, dk) \
            or tuple(v.shape) != (B, H, dv) or tuple(o.shape) != (B, H, dv):
        raise ValueError("shape mismatch")
    st = load_library().la_decode_step(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       o.data_ptr(), B, H, dk, dv, float(eps), _dtype_code(q),
                                       _stream_ptr(stream))
    _check("la_decode_step", st)
    return o


def _gamma_tensor(gamma, H: int):
    import torch
    _need_cuda(gamma)
    if gamma.dtype != torch.float32 or tuple(gamma.shape) != (H,):
        raise ValueError("gamma must be a float32 tensor of shape [H]")


def la_forward_causal_decay(q, k, v, gamma, o=None, chunk: int = 128, eps: float = 1e-6, stream=None):
    """Causal forward with a decayed state, gamma [H] fp32 (one decay per head);
    q, k [B,H,N,dk], v [B,H,N,dv]; returns o [B,H,N,dv]."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, N, dk) or tuple(v.shape[:-1]) != (B, H, N) or tuple(o.shape) != (B, H, N, dv):
        raise ValueError("shape mismatch")
    _gamma_tensor(gamma, H)
    st = load_library().la_forward_causal_decay(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                gamma.data_ptr(), B, H, N, dk, dv, int(chunk), float(eps),
                                                _dtype_code(q), _stream_ptr(stream))
    _check("la_forward_causal_decay", st)
    return o


def la_decode_step_decay(S, z, q, k, v, gamma, o=None, eps: float = 1e-6, stream=None):
    """One decayed decode step (S = g S + phi(k) v^T, z = g z + phi(k), g = gamma[h]);
    S, z updated in place; returns o [B,H,dv]."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(S, z, q, k, v, o)
    _same_dtype(q, k, v, o)
    if S.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("S and z must be float32")
    B, H, dk = q.shape
    dv = v.shape[-1]
    if tuple(S.shape) != (B, H, dk, dv) or tuple(z.shape) != (B, H, dk) or tuple(k.shape) != (B, H, dk) \
            or tuple(v.shape) != (B, H, dv) or tuple(o.shape) != (B, H, dv):
        raise ValueError("shape mismatch")
    _gamma_tensor(gamma, H)
    st = load_library().la_decode_step_decay(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(),
                                             v.data_ptr(), o.data_ptr(), gamma.data_ptr(), B, H, dk, dv,
                                             float(eps), _dtype_code(q), _stream_ptr(stream))
    _check("la_decode_step_decay", st)
    return o


def la_prefill_state(k, v, S=None, z=None, stream=None):
    """S = sum_t phi(k_t) v_t^T, z = sum_t phi(k_t) over N tokens; returns (S, z) fp32."""
    import torch
    B, H, N, dk = k.shape
    dv = v.shape[-1]
    if S is None:
        S = torch.empty((B, H, dk, dv), dtype=torch.float32, device=k.device)
    if z is None:
        z = torch.empty((B, H, dk), dtype=torch.float32, device=k.device)
    _need_cuda(k, v, S, z)
    _same_dtype(k, v)
    if tuple(v.shape[:-1]) != (B, H, N) or tuple(S.shape) != (B, H, dk, dv) or tuple(z.shape) != (B, H, dk):
        raise ValueError("shape mismatch")
    st = load_library().la_prefill_state(k.data_ptr(), v.data_ptr(), S.data_ptr(), z.data_ptr(),
                                         B, H, N, dk, dv, _dtype_code(k), _stream_ptr(stream))
    _check("la_prefill_state", st)
    return S, z


def la_prefill_state_decay(k, v, gamma, S=None, z=None, stream=None):
    """Decayed prefix state: S = sum_t g^(N-1-t) phi(k_t) v_t^T, z likewise, g = gamma[h];
    returns (S, z) fp32."""
    import torch
    B, H, N, dk = k.shape
    dv = v.shape[-1]
    if S is None:
        S = torch.empty((B, H, dk, dv), dtype=torch.float32, device=k.device)
    if z is None:
        z = torch.empty((B, H, dk), dtype=torch.float32, device=k.device)
    _need_cuda(k, v, S, z)
    _same_dtype(k, v)
    if tuple(v.shape[:-1]) != (B, H, N) or tuple(S.shape) != (B, H, dk, dv) or tuple(z.shape) != (B, H, dk):
        raise ValueError("shape mismatch")
    _gamma_tensor(gamma, H)
    st = load_library().la_prefill_state_decay(k.data_ptr(), v.data_ptr(), gamma.data_ptr(), S.data_ptr(),
                                               z.data_ptr(), B, H, N, dk, dv, _dtype_code(k), _stream_ptr(stream))
    _check("la_prefill_state_decay", st)
    return S, z


def _alpha_tensor(alpha, shape):
    import torch
    if not isinstance(alpha, torch.Tensor) or alpha.dtype != torch.float32 or not alpha.is_cuda \
            or not alpha.is_contiguous() or tuple(alpha.shape) != tuple(shape):
        raise ValueError("alpha must be a contiguous float32 CUDA tensor of shape %s" % (tuple(shape),))


def la_forward_causal_gated(q, k, v, alpha, o=None, eps: float = 1e-6, stream=None):
    """Causal forward with a gated state, one gate per key feature: alpha [B,H,N,dk]
    fp32 (S_t = Diag(alpha_t) S_{t-1} + phi(k_t) v_t^T, z alike); returns o [B,H,N,dv]."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, N, dk) or tuple(v.shape[:-1]) != (B, H, N) or tuple(o.shape) != (B, H, N, dv):
        raise ValueError("shape mismatch")
    _alpha_tensor(alpha, k.shape)
    st = load_library().la_forward_causal_gated(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                alpha.data_ptr(), B, H, N, dk, dv, float(eps), _dtype_code(q),
                                                _stream_ptr(stream))
    _check("la_forward_causal_gated", st)
    return o


def la_prefill_state_gated(k, v, alpha, S=None, z=None, stream=None):
    """State after the gated recurrence over N tokens from zero; returns (S, z) fp32."""
    import torch
    B, H, N, dk = k.shape
    dv = v.shape[-1]
    if S is None:
        S = torch.empty((B, H, dk, dv), dtype=torch.float32, device=k.device)
    if z is None:
        z = torch.empty((B, H, dk), dtype=torch.float32, device=k.device)
    _need_cuda(k, v, S, z)
    _same_dtype(k, v)
    if tuple(v.shape[:-1]) != (B, H, N) or tuple(S.shape) != (B, H, dk, dv) or tuple(z.shape) != (B, H, dk):
        raise ValueError("shape mismatch")
    _alpha_tensor(alpha, k.shape)
    st = load_library().la_prefill_state_gated(k.data_ptr(), v.data_ptr(), alpha.data_ptr(), S.data_ptr(),
                                               z.data_ptr(), B, H, N, dk, dv, _dtype_code(k), _stream_ptr(stream))
    _check("la_prefill_state_gated", st)
    return S, z


def la_decode_step_gated(S, z, q, k, v, alpha, o=None, eps: float = 1e-6, stream=None):
    """One gated decode step in place; q, k, alpha [B,H,dk], v [B,H,dv]; returns o [B,H,dv]."""
    import torch
    if o is None:
        o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    _need_cuda(S, z, q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, dk = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, dk) or tuple(v.shape) != (B, H, dv) or tuple(S.shape) != (B, H, dk, dv) \
            or tuple(z.shape) != (B, H, dk):
        raise ValueError("shape mismatch")
    _alpha_tensor(alpha, k.shape)
    st = load_library().la_decode_step_gated(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             o.data_ptr(), alpha.data_ptr(), B, H, dk, dv, float(eps),
                                             _dtype_code(q), _stream_ptr(stream))
    _check("la_decode_step_gated", st)
    return o


def _gamma_ptr(gamma, H):
    if gamma is None:
        return None
    _gamma_tensor(gamma, H)
    return gamma.data_ptr()


def la_forward_causal_ex(q, k, v, o=None, gamma=None, feature_map="elu1", shift=0.0, normalize=True,
                         chunk: int = 128, eps: float = 1e-6, stream=None):
    """Causal forward with a feature map ("elu1", "relu": max(x, 0) + shift, "identity":
    x + shift), with or without the normaliser, with or without a per-head decay gamma [H]."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, N, dk) or tuple(v.shape[:-1]) != (B, H, N) or tuple(o.shape) != (B, H, N, dv):
        raise ValueError("shape mismatch")
    st = load_library().la_forward_causal_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                             _gamma_ptr(gamma, H), _variant(feature_map, shift, normalize),
                                             B, H, N, dk, dv, int(chunk), float(eps), _dtype_code(q),
                                             _stream_ptr(stream))
    _check("la_forward_causal_ex", st)
    return o


def la_forward_noncausal_ex(q, k, v, o=None, feature_map="elu1", shift=0.0, normalize=True, eps: float = 1e-6,
                            stream=None):
    """Non-causal forward with a feature map, with or without the normaliser."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, N, dk) or tuple(v.shape[:-1]) != (B, H, N) or tuple(o.shape) != (B, H, N, dv):
        raise ValueError("shape mismatch")
    st = load_library().la_forward_noncausal_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                _variant(feature_map, shift, normalize), B, H, N, dk, dv,
                                                float(eps), _dtype_code(q), _stream_ptr(stream))
    _check("la_forward_noncausal_ex", st)
    return o


def la_decode_step_ex(S, z, q, k, v, o=None, gamma=None, feature_map="elu1", shift=0.0, normalize=True,
                      eps: float = 1e-6, stream=None):
    """One decode step with a feature map, normaliser choice and optional decay; S, z in place."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(S, z, q, k, v, o)
    _same_dtype(q, k, v, o)
    if S.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("S and z must be float32")
    B, H, dk = q.shape
    dv = v.shape[-1]
    if tuple(S.shape) != (B, H, dk, dv) or tuple(z.shape) != (B, H, dk) or tuple(k.shape) != (B, H, dk) \
            or tuple(v.shape) != (B, H, dv) or tuple(o.shape) != (B, H, dv):
        raise ValueError("shape mismatch")
    st = load_library().la_decode_step_ex(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          o.data_ptr(), _gamma_ptr(gamma, H), _variant(feature_map, shift, normalize),
                                          B, H, dk, dv, float(eps), _dtype_code(q), _stream_ptr(stream))
    _check("la_decode_step_ex", st)
    return o


def la_prefill_state_ex(k, v, S=None, z=None, gamma=None, feature_map="elu1", shift=0.0, stream=None):
    """Prefix state under a feature map and an optional decay; returns (S, z) fp32."""
    import torch
    B, H, N, dk = k.shape
    dv = v.shape[-1]
    if S is None:
        S = torch.empty((B, H, dk, dv), dtype=torch.float32, device=k.device)
    if z is None:
        z = torch.empty((B, H, dk), dtype=torch.float32, device=k.device)
    _need_cuda(k, v, S, z)
    _same_dtype(k, v)
    if tuple(v.shape[:-1]) != (B, H, N) or tuple(S.shape) != (B, H, dk, dv) or tuple(z.shape) != (B, H, dk):
        raise ValueError("shape mismatch")
    st = load_library().la_prefill_state_ex(k.data_ptr(), v.data_ptr(), _gamma_ptr(gamma, H),
                                            _variant(feature_map, shift, True), S.data_ptr(), z.data_ptr(),
                                            B, H, N, dk, dv, _dtype_code(k), _stream_ptr(stream))
    _check("la_prefill_state_ex", st)
    return S, z


def la_backward_causal(q, k, v, dout, dq=None, dk=None, dv=None, eps: float = 1e-6, stream=None):
    """Gradients (dq, dk, dv) of sum(dout * o) for the causal forward (elu + 1, normalised)."""
    import torch
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need_cuda(q, k, v, dout, dq, dk, dv)
    _same_dtype(q, k, v, dout, dq, dk, dv)
    B, H, N, d_k = q.shape
    d_v = v.shape[-1]
    if tuple(k.shape) != (B, H, N, d_k) or tuple(v.shape[:-1]) != (B, H, N) or tuple(dout.shape) != tuple(v.shape) \
            or tuple(dq.shape) != tuple(q.shape) or tuple(dk.shape) != tuple(k.shape) or tuple(dv.shape) != tuple(v.shape):
        raise ValueError("shape mismatch")
    st = load_library().la_backward_causal(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(), dq.data_ptr(),
                                           dk.data_ptr(), dv.data_ptr(), B, H, N, d_k, d_v, float(eps),
                                           _dtype_code(q), _stream_ptr(stream))
    _check("la_backward_causal", st)
    return dq, dk, dv


def _favor_w(w, x, d):
    _need_cuda(w)
    if w.dim() != 2 or w.shape[1] != d or w.dtype != x.dtype:
        raise ValueError("w must be [m, d] with the dtype of the inputs")
    return w.shape[0]


def la_favor_features(x, w, phi=None, stream=None):
    """FAVOR+ features phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m); x [B,H,N,d], w [m,d];
    returns phi [B,H,N,m] in the dtype of x."""
    import torch
    B, H, N, d = x.shape
    m = _favor_w(w, x, d)
    if phi is None:
        phi = torch.empty((B, H, N, m), dtype=x.dtype, device=x.device)
    _need_cuda(x, phi)
    _same_dtype(x, w, phi)
    if tuple(phi.shape) != (B, H, N, m):
        raise ValueError("shape mismatch")
    st = load_library().la_favor_features(x.data_ptr(), w.data_ptr(), phi.data_ptr(), B, H, N, d, m,
                                          _dtype_code(x), _stream_ptr(stream))
    _check("la_favor_features", st)
    return phi


def _favor_shapes(q, k, v, o, w):
    _need_cuda(q, k, v, o)
    _same_dtype(q, k, v, o)
    B, H, N, d = q.shape
    dv = v.shape[-1]
    if tuple(k.shape) != (B, H, N, d) or tuple(v.shape[:-1]) != (B, H, N) or tuple(o.shape) != (B, H, N, dv):
        raise ValueError("shape mismatch")
    return B, H, N, d, dv, _favor_w(w, q, d)


def la_forward_causal_favor(q, k, v, w, o=None, chunk: int = 128, eps: float = 1e-6, stream=None):
    """Causal linear attention on FAVOR+ features of q and k (projections w [m, d])."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    B, H, N, d, dv, m = _favor_shapes(q, k, v, o, w)
    st = load_library().la_forward_causal_favor(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                w.data_ptr(), B, H, N, d, dv, m, int(chunk), float(eps),
                                                _dtype_code(q), _stream_ptr(stream))
    _check("la_forward_causal_favor", st)
    return o


def la_forward_noncausal_favor(q, k, v, w, o=None, eps: float = 1e-6, stream=None):
    """Non-causal linear attention on FAVOR+ features of q and k (projections w [m, d])."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    B, H, N, d, dv, m = _favor_shapes(q, k, v, o, w)
    st = load_library().la_forward_noncausal_favor(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                   w.data_ptr(), B, H, N, d, dv, m, float(eps), _dtype_code(q),
                                                   _stream_ptr(stream))
    _check("la_forward_noncausal_favor", st)
    return o


def la_prefill_state_favor(k, v, w, S=None, z=None, stream=None):
    """Prefix state on FAVOR+ features of k (projections w [m, d]); returns (S [B,H,m,dv], z [B,H,m]) fp32."""
    import torch
    B, H, N, d = k.shape
    dv = v.shape[-1]
    m = _favor_w(w, k, d)
    if S is None:
        S = torch.empty((B, H, m, dv), dtype=torch.float32, device=k.device)
    if z is None:
        z = torch.empty((B, H, m), dtype=torch.float32, device=k.device)
    _need_cuda(k, v, S, z)
    _same_dtype(k, v)
    if tuple(v.shape[:-1]) != (B, H, N) or tuple(S.shape) != (B, H, m, dv) or tuple(z.shape) != (B, H, m):
        raise ValueError("shape mismatch")
    st = load_library().la_prefill_state_favor(k.data_ptr(), v.data_ptr(), w.data_ptr(), S.data_ptr(), z.data_ptr(),
                                               B, H, N, d, dv, m, _dtype_code(k), _stream_ptr(stream))
    _check("la_prefill_state_favor", st)
    return S, z


def la_decode_step_favor(S, z, q, k, v, w, o=None, eps: float = 1e-6, stream=None):
    """One decode step on FAVOR+ features of q and k; S [B,H,m,dv], z [B,H,m] fp32 updated in place."""
    import torch
    if o is None:
        o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _need_cuda(S, z, q, k, v, o)
    _same_dtype(q, k, v, o)
    if S.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("S and z must be float32")
    B, H, d = q.shape
    dv = v.shape[-1]
    m = _favor_w(w, q, d)
    if tuple(S.shape) != (B, H, m, dv) or tuple(z.shape) != (B, H, m) or tuple(k.shape) != (B, H, d) \
            or tuple(v.shape) != (B, H, dv) or tuple(o.shape) != (B, H, dv):
        raise ValueError("shape mismatch")
    st = load_library().la_decode_step_favor(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             o.data_ptr(), w.data_ptr(), B, H, d, dv, m, float(eps), _dtype_code(q),
                                             _stream_ptr(stream))
    _check("la_decode_step_favor", st)
    return o


def la_get_device_status(stream=None) -> int:
    return load_library().la_get_device_status(_stream_ptr(stream))


def la_status_string(status: int) -> str:
    return load_library().la_status_string(int(status)).decode()


def la_last_cuda_error() -> int:
    return load_library().la_last_cuda_error()


def la_version() -> int:
    return load_library().la_version()


def la_kernel_launches() -> int:
    return int(load_library().la_kernel_launches())
