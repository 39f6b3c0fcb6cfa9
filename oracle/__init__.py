"""Float64 CPU oracle for causal kernelized (linear) attention, phi = elu + 1.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the benchmark's CPU-baseline / reference arm may import
this package.  It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``la_oracle.c`` (plain double-precision loops, one
(batch, head) sequence at a time, OpenMP across sequences).  This module only
compiles it with gcc and marshals numpy arrays through ctypes.

Inputs may be float64, float32, or uint16 arrays holding bf16 bit patterns;
they are widened exactly inside the C code.  Shapes: q, k [..., N, dk],
v [..., N, dv] with identical leading dims; outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblaoracle.so")
_lock = threading.Lock()
_lib = None

_TYPE_CODE = {np.dtype(np.float64): 0, np.dtype(np.float32): 1, np.dtype(np.uint16): 2}


def build(force: bool = False, out_path: str = _LIB_PATH, defines=()) -> str:
    """Compile la_oracle.c into a shared library (gcc, -O3, no fast-math).

    ``-ffp-contract=off`` keeps results identical on x86-64 and aarch64 (no
    fused multiply-add contraction).  ``defines`` is for tests that compile a
    deliberately wrong variant to show the pins catch it.
    """
    if not force and not defines and os.path.exists(out_path) and \
            os.path.getmtime(out_path) >= os.path.getmtime(_SRC):
        return out_path
    cmd = ["gcc", "-O3", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
           "-shared", "-std=c11", "-Wall", "-Wno-unknown-pragmas", _SRC, "-o", out_path, "-lm"]
    cmd[1:1] = ["-D" + d for d in defines]
    tmp = out_path + ".tmp%d" % os.getpid()
    cmd[cmd.index(out_path)] = tmp
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _declare(lib):
    P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    sigs = {
        "la_oracle_phi": ([D], D),
        "la_oracle_causal_recurrent": ([P, P, P, I, P, I, I, I, I, D], None),
        "la_oracle_causal_chunked": ([P, P, P, I, P, I, I, I, I, I, D], None),
        "la_oracle_causal_quadratic": ([P, P, P, I, P, I, I, I, I, D], None),
        "la_oracle_prefill_state": ([P, P, I, P, P, I, I, I, I], None),
        "la_oracle_noncausal": ([P, P, P, I, P, I, I, I, I, D], None),
        "la_oracle_noncausal_pairwise": ([P, P, P, I, P, I, I, I, I, D], None),
        "la_oracle_decode_step": ([P, P, P, P, P, I, P, I, I, I, D], None),
        "la_oracle_causal_decay_recurrent": ([P, P, P, I, P, P, I, I, I, I, D], None),
        "la_oracle_causal_decay_quadratic": ([P, P, P, I, P, P, I, I, I, I, D], None),
        "la_oracle_decode_step_decay": ([P, P, P, P, P, I, P, P, I, I, I, D], None),
        "la_oracle_causal_general": ([P, P, P, I, P, I, D, I, P, I, I, I, I, D], None),
        "la_oracle_causal_general_quadratic": ([P, P, P, I, P, I, D, I, P, I, I, I, I, D], None),
        "la_oracle_prefill_state_general": ([P, P, I, P, I, D, P, P, I, I, I, I], None),
        "la_oracle_noncausal_general": ([P, P, P, I, I, D, I, P, I, I, I, I, D], None),
        "la_oracle_decode_step_general": ([P, P, P, P, P, I, P, I, D, I, P, I, I, I, D], None),
        "la_oracle_causal_backward": ([P, P, P, P, I, P, P, P, I, I, I, I, D], None),
        "la_oracle_favor_features": ([P, I, P, P, ctypes.c_longlong, I, I], None),
        "la_oracle_causal_gated_recurrent": ([P, P, P, I, P, P, I, I, I, I, D], None),
        "la_oracle_causal_gated_quadratic": ([P, P, P, I, P, P, I, I, I, I, D], None),
        "la_oracle_decode_step_gated": ([P, P, P, P, P, I, P, P, I, I, I, D], None),
        "la_oracle_prefill_state_gated": ([P, P, I, P, P, P, I, I, I, I], None),
        "la_oracle_num_threads": ([], I),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load(path: str = None):
    """Build (if needed) and load the oracle library; returns the ctypes handle."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _prep(*arrays):
    t = None
    out = []
    for a in arrays:
        a = np.ascontiguousarray(a)
        if a.dtype not in _TYPE_CODE:
            a = np.ascontiguousarray(a, dtype=np.float64)
        if t is None:
            t = a.dtype
        elif a.dtype != t:
            raise TypeError("q, k, v must share one element type")
        out.append(a)
    return out, _TYPE_CODE[t]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """Bound oracle functions; ``lib`` may be a deliberately wrong test build."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def phi(self, x: float) -> float:
        return self.lib.la_oracle_phi(float(x))

    def num_threads(self) -> int:
        return self.lib.la_oracle_num_threads()

    def _fwd(self, fname, q, k, v, eps, *extra):
        (q, k, v), t = _prep(q, k, v)
        N, dk = q.shape[-2], q.shape[-1]
        dv = v.shape[-1]
        lead = q.shape[:-2]
        if k.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
            raise ValueError("shape mismatch")
        BH = int(np.prod(lead)) if lead else 1
        o = np.empty(lead + (N, dv), dtype=np.float64)
        if BH and N and dv:
            fn = getattr(self.lib, fname)
            if extra:
                fn(_ptr(q), _ptr(k), _ptr(v), t, _ptr(o), BH, N, dk, dv, *extra, float(eps))
            else:
                fn(_ptr(q), _ptr(k), _ptr(v), t, _ptr(o), BH, N, dk, dv, float(eps))
        return o

    def causal_recurrent(self, q, k, v, eps=1e-6):
        return self._fwd("la_oracle_causal_recurrent", q, k, v, eps)

    def causal_chunked(self, q, k, v, chunk, eps=1e-6):
        return self._fwd("la_oracle_causal_chunked", q, k, v, eps, int(chunk))

    def causal_quadratic(self, q, k, v, eps=1e-6):
        return self._fwd("la_oracle_causal_quadratic", q, k, v, eps)

    def noncausal(self, q, k, v, eps=1e-6):
        return self._fwd("la_oracle_noncausal", q, k, v, eps)

    def noncausal_pairwise(self, q, k, v, eps=1e-6):
        return self._fwd("la_oracle_noncausal_pairwise", q, k, v, eps)

    def prefill_state(self, k, v):
        """S [..., dk, dv] and z [..., dk] summed over all N tokens."""
        (k, v), t = _prep(k, v)
        N, dk, dv = k.shape[-2], k.shape[-1], v.shape[-1]
        lead = k.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        S = np.zeros(lead + (dk, dv), dtype=np.float64)
        z = np.zeros(lead + (dk,), dtype=np.float64)
        if BH:
            self.lib.la_oracle_prefill_state(_ptr(k), _ptr(v), t, _ptr(S), _ptr(z), BH, N, dk, dv)
        return S, z

    def decode_step(self, S, z, q, k, v, eps=1e-6):
        """One step for every head: updates float64 S [...,dk,dv], z [...,dk] in place.

        q, k [..., dk], v [..., dv]; returns o [..., dv] float64.
        """
        if S.dtype != np.float64 or z.dtype != np.float64 or not S.flags.c_contiguous \
                or not z.flags.c_contiguous:
            raise TypeError("S and z must be C-contiguous float64 (updated in place)")
        (q, k, v), t = _prep(q, k, v)
        dk, dv = q.shape[-1], v.shape[-1]
        lead = q.shape[:-1]
        BH = int(np.prod(lead)) if lead else 1
        if S.shape != lead + (dk, dv) or z.shape != lead + (dk,):
            raise ValueError("state shape mismatch")
        o = np.empty(lead + (dv,), dtype=np.float64)
        if BH:
            self.lib.la_oracle_decode_step(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v), t,
                                           _ptr(o), BH, dk, dv, float(eps))
        return o


    # ---------------------------------------------------------------- decayed state
    @staticmethod
    def _gamma(gamma, lead):
        g = np.ascontiguousarray(np.broadcast_to(np.asarray(gamma, dtype=np.float64), lead)).reshape(-1)
        if np.any(g < 0) or np.any(g > 1) or not np.all(np.isfinite(g)):
            raise ValueError("gamma must lie in [0, 1]")
        return np.ascontiguousarray(g)

    def _fwd_decay(self, fname, q, k, v, gamma, eps):
        (q, k, v), t = _prep(q, k, v)
        N, dk = q.shape[-2], q.shape[-1]
        dv = v.shape[-1]
        lead = q.shape[:-2]
        if k.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
            raise ValueError("shape mismatch")
        g = self._gamma(gamma, lead)
        BH = int(np.prod(lead)) if lead else 1
        o = np.empty(lead + (N, dv), dtype=np.float64)
        if BH and N and dv:
            getattr(self.lib, fname)(_ptr(q), _ptr(k), _ptr(v), t, _ptr(g), _ptr(o), BH, N, dk, dv, float(eps))
        return o

    def causal_decay_recurrent(self, q, k, v, gamma, eps=1e-6):
        """Decayed causal form; gamma broadcasts to the leading dims ([H] per head)."""
        return self._fwd_decay("la_oracle_causal_decay_recurrent", q, k, v, gamma, eps)

    def causal_decay_quadratic(self, q, k, v, gamma, eps=1e-6):
        return self._fwd_decay("la_oracle_causal_decay_quadratic", q, k, v, gamma, eps)

    def decode_step_decay(self, S, z, q, k, v, gamma, eps=1e-6):
        """One decayed step for every head, S and z (float64) updated in place."""
        if S.dtype != np.float64 or z.dtype != np.float64 or not S.flags.c_contiguous \
                or not z.flags.c_contiguous:
            raise TypeError("S and z must be C-contiguous float64 (updated in place)")
        (q, k, v), t = _prep(q, k, v)
        dk, dv = q.shape[-1], v.shape[-1]
        lead = q.shape[:-1]
        BH = int(np.prod(lead)) if lead else 1
        if S.shape != lead + (dk, dv) or z.shape != lead + (dk,):
            raise ValueError("state shape mismatch")
        g = self._gamma(gamma, lead)
        o = np.empty(lead + (dv,), dtype=np.float64)
        if BH:
            self.lib.la_oracle_decode_step_decay(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v), t, _ptr(g),
                                                 _ptr(o), BH, dk, dv, float(eps))
        return o

    # ------------------------------------------------ feature maps and the normaliser
    # fmap: 0 = elu + 1, 1 = max(x, 0) + shift, 2 = x + shift; normalize: divide by
    # max(phi(q)^T z, eps) or not; gamma: None (no decay) or broadcast to the heads.
    FMAPS = {"elu1": 0, "relu": 1, "identity": 2}

    def _gptr(self, gamma, lead):
        if gamma is None:
            return None, None
        g = self._gamma(gamma, lead)
        return g, _ptr(g)

    def _fwd_general(self, fname, q, k, v, gamma, fmap, shift, normalize, eps):
        (q, k, v), t = _prep(q, k, v)
        N, dk = q.shape[-2], q.shape[-1]
        dv = v.shape[-1]
        lead = q.shape[:-2]
        if k.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
            raise ValueError("shape mismatch")
        g, gp = self._gptr(gamma, lead)
        BH = int(np.prod(lead)) if lead else 1
        o = np.empty(lead + (N, dv), dtype=np.float64)
        if BH and N and dv:
            getattr(self.lib, fname)(_ptr(q), _ptr(k), _ptr(v), t, gp, self.FMAPS[fmap], float(shift),
                                     int(bool(normalize)), _ptr(o), BH, N, dk, dv, float(eps))
        return o

    def causal_general(self, q, k, v, gamma=None, fmap="elu1", shift=0.0, normalize=True, eps=1e-6):
        """The causal recurrence with a feature map, an optional decay and an optional normaliser."""
        return self._fwd_general("la_oracle_causal_general", q, k, v, gamma, fmap, shift, normalize, eps)

    def causal_general_quadratic(self, q, k, v, gamma=None, fmap="elu1", shift=0.0, normalize=True,
                                 eps=1e-6):
        return self._fwd_general("la_oracle_causal_general_quadratic", q, k, v, gamma, fmap, shift,
                                 normalize, eps)

    def noncausal_general(self, q, k, v, fmap="elu1", shift=0.0, normalize=True, eps=1e-6):
        (q, k, v), t = _prep(q, k, v)
        N, dk = q.shape[-2], q.shape[-1]
        dv = v.shape[-1]
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        o = np.empty(lead + (N, dv), dtype=np.float64)
        if BH and N and dv:
            self.lib.la_oracle_noncausal_general(_ptr(q), _ptr(k), _ptr(v), t, self.FMAPS[fmap], float(shift),
                                                 int(bool(normalize)), _ptr(o), BH, N, dk, dv, float(eps))
        return o

    def prefill_state_general(self, k, v, gamma=None, fmap="elu1", shift=0.0):
        (k, v), t = _prep(k, v)
        N, dk, dv = k.shape[-2], k.shape[-1], v.shape[-1]
        lead = k.shape[:-2]
        g, gp = self._gptr(gamma, lead)
        BH = int(np.prod(lead)) if lead else 1
        S = np.zeros(lead + (dk, dv), dtype=np.float64)
        z = np.zeros(lead + (dk,), dtype=np.float64)
        if BH:
            self.lib.la_oracle_prefill_state_general(_ptr(k), _ptr(v), t, gp, self.FMAPS[fmap], float(shift),
                                                     _ptr(S), _ptr(z), BH, N, dk, dv)
        return S, z

    def decode_step_general(self, S, z, q, k, v, gamma=None, fmap="elu1", shift=0.0, normalize=True,
                            eps=1e-6):
        if S.dtype != np.float64 or z.dtype != np.float64 or not S.flags.c_contiguous \
                or not z.flags.c_contiguous:
            raise TypeError("S and z must be C-contiguous float64 (updated in place)")
        (q, k, v), t = _prep(q, k, v)
        dk, dv = q.shape[-1], v.shape[-1]
        lead = q.shape[:-1]
        BH = int(np.prod(lead)) if lead else 1
        if S.shape != lead + (dk, dv) or z.shape != lead + (dk,):
            raise ValueError("state shape mismatch")
        g, gp = self._gptr(gamma, lead)
        o = np.empty(lead + (dv,), dtype=np.float64)
        if BH:
            self.lib.la_oracle_decode_step_general(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v), t, gp,
                                                   self.FMAPS[fmap], float(shift), int(bool(normalize)),
                                                   _ptr(o), BH, dk, dv, float(eps))
        return o

    # ---------------------------------------------------------------- gated state
    # alpha: the per-key gate, one value in [0, 1] per (token, key feature), shaped
    # like k ([..., N, dk]; [..., dk] for a decode step).
    @staticmethod
    def _alpha(alpha, shape):
        a = np.ascontiguousarray(np.broadcast_to(np.asarray(alpha, dtype=np.float64), shape))
        if np.any(a < 0) or np.any(a > 1) or not np.all(np.isfinite(a)):
            raise ValueError("alpha must lie in [0, 1]")
        return a

    def _fwd_gated(self, fname, q, k, v, alpha, eps):
        (q, k, v), t = _prep(q, k, v)
        N, dk = q.shape[-2], q.shape[-1]
        dv = v.shape[-1]
        lead = q.shape[:-2]
        if k.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
            raise ValueError("shape mismatch")
        a = self._alpha(alpha, k.shape)
        BH = int(np.prod(lead)) if lead else 1
        o = np.empty(lead + (N, dv), dtype=np.float64)
        if BH and N and dv:
            getattr(self.lib, fname)(_ptr(q), _ptr(k), _ptr(v), t, _ptr(a), _ptr(o), BH, N, dk, dv, float(eps))
        return o

    def causal_gated_recurrent(self, q, k, v, alpha, eps=1e-6):
        """Gated causal form: S_t = Diag(alpha_t) S_{t-1} + phi(k_t) v_t^T, z likewise."""
        return self._fwd_gated("la_oracle_causal_gated_recurrent", q, k, v, alpha, eps)

    def causal_gated_quadratic(self, q, k, v, alpha, eps=1e-6):
        return self._fwd_gated("la_oracle_causal_gated_quadratic", q, k, v, alpha, eps)

    def decode_step_gated(self, S, z, q, k, v, alpha, eps=1e-6):
        """One gated step for every head, S and z (float64) updated in place; alpha [..., dk]."""
        if S.dtype != np.float64 or z.dtype != np.float64 or not S.flags.c_contiguous \
                or not z.flags.c_contiguous:
            raise TypeError("S and z must be C-contiguous float64 (updated in place)")
        (q, k, v), t = _prep(q, k, v)
        dk, dv = q.shape[-1], v.shape[-1]
        lead = q.shape[:-1]
        BH = int(np.prod(lead)) if lead else 1
        if S.shape != lead + (dk, dv) or z.shape != lead + (dk,):
            raise ValueError("state shape mismatch")
        a = self._alpha(alpha, k.shape)
        o = np.empty(lead + (dv,), dtype=np.float64)
        if BH:
            self.lib.la_oracle_decode_step_gated(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v), t, _ptr(a),
                                                 _ptr(o), BH, dk, dv, float(eps))
        return o

    def prefill_state_gated(self, k, v, alpha):
        """S [..., dk, dv], z [..., dk] after the gated recurrence over all N tokens."""
        (k, v), t = _prep(k, v)
        N, dk, dv = k.shape[-2], k.shape[-1], v.shape[-1]
        lead = k.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        a = self._alpha(alpha, k.shape)
        S = np.zeros(lead + (dk, dv), dtype=np.float64)
        z = np.zeros(lead + (dk,), dtype=np.float64)
        if BH:
            self.lib.la_oracle_prefill_state_gated(_ptr(k), _ptr(v), t, _ptr(a), _ptr(S), _ptr(z), BH, N, dk, dv)
        return S, z

    # ---------------------------------------------------------------- backward pass
    def causal_backward(self, q, k, v, dout, eps=1e-6):
        """Gradients (dq, dk, dv) of sum(dout * o) for the causal form (elu + 1, normalised)."""
        (q, k, v, dout), t = _prep(q, k, v, dout)
        N, dk = q.shape[-2], q.shape[-1]
        dv = v.shape[-1]
        lead = q.shape[:-2]
        if k.shape != q.shape or v.shape[:-1] != q.shape[:-1] or dout.shape != v.shape:
            raise ValueError("shape mismatch")
        BH = int(np.prod(lead)) if lead else 1
        gq = np.zeros(q.shape, dtype=np.float64)
        gk = np.zeros(k.shape, dtype=np.float64)
        gv = np.zeros(v.shape, dtype=np.float64)
        if BH and N:
            self.lib.la_oracle_causal_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), t, _ptr(gq), _ptr(gk), _ptr(gv),
                                               BH, N, dk, dv, float(eps))
        return gq, gk, gv

    # ---------------------------------------------------------------- FAVOR+ features
    def favor_features(self, x, W):
        """phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m) for x [..., d], W [m, d]; returns [..., m]."""
        (x,), t = _prep(x)
        W = np.ascontiguousarray(W, dtype=np.float64)
        m, d = W.shape
        if x.shape[-1] != d:
            raise ValueError("shape mismatch")
        rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
        out = np.empty(x.shape[:-1] + (m,), dtype=np.float64)
        if rows:
            self.lib.la_oracle_favor_features(_ptr(x), t, _ptr(W), _ptr(out), rows, d, m)
        return out

    def causal_favor(self, q, k, v, W, eps=1e-6):
        """Causal linear attention on FAVOR+ features (the identity map on phi(q), phi(k))."""
        return self.causal_general(self.favor_features(q, W), self.favor_features(k, W), np.asarray(v, np.float64)
                                   if np.asarray(v).dtype != np.uint16 else _widen_bf16(v), fmap="identity",
                                   shift=0.0, normalize=True, eps=eps)


    def noncausal_favor(self, q, k, v, W, eps=1e-6):
        """Non-causal linear attention on FAVOR+ features (the identity map on phi(q), phi(k))."""
        return self.noncausal_general(self.favor_features(q, W), self.favor_features(k, W),
                                      np.asarray(v, np.float64) if np.asarray(v).dtype != np.uint16
                                      else _widen_bf16(v), fmap="identity", shift=0.0, normalize=True, eps=eps)

def _widen_bf16(bits):
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


_default = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
