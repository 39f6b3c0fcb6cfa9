"""The method's edge cases on every GPU path, element by element against the
float64 oracle (needs a GB300).

  * The clamp of the denominator binds.  The output is
    phi(q)^T S / max(phi(q)^T z, eps) ("Linear Attention", the chunked listing's
    clamp(min=1e-6); "26. Linear (Kernelized) Attention", Step-by-Step step 6).
    With eps = 1e8 it binds on every row; with eps = 1e4 on the early rows of a
    causal sequence only, so one launch takes both branches.  Queries pushed to
    -30 (phi(q) = exp(-30) ~ 1e-13) make it bind at eps = 1e-6.
  * Inputs well outside N(0, 1): sigma = 2 and 4 on the tensor-core paths, where
    phi's exponential sees |x| up to ~20.
  * The first output equals the first value, o_0 = v_0, exactly (bf16: the
    operand P_00 is the same rounded number in the numerator and the normaliser).
  * The identity feature map with the normaliser, at a shift that keeps every
    phi positive (where that form is well defined).

A clamped output is tiny (|o| ~ |v| * phi(q).z / eps), so besides the absolute
bf16 bounds (max 2e-2, mean 2e-3) every case here is held to a normwise bound,
max|gpu - oracle| / max|oracle|: 1e-5 for fp32 inputs, 2e-2 for bf16.

Inputs drawn at sigma > 1 give outputs sigma times larger (o is a convex
combination of the v_j), and a bf16 output carries its own rounding, up to
|o| * 2^-9 (0.0156 at |o| = 6, 0.03 at |o| = 12): there the absolute bounds are
scaled by sigma (max 2e-2 * sigma, mean 2e-3 * sigma) and the normwise bound of
2e-2 holds as it is.
"""
import numpy as np
import pytest

import workloads
from gpu_util import assert_parity, errors, from_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NORMWISE = {"f32": 1e-5, "bf16": 2e-2}


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


def check(got, ref, dtype, what):
    e = assert_parity(got, ref, dtype, what)
    assert e["normwise"] <= NORMWISE[dtype], (what, e)
    return e


def check_scaled(got, ref, sigma, what):
    """bf16 outputs of inputs drawn at scale sigma (see the module docstring)."""
    e = errors(got, ref)
    assert e["finite"], what
    assert e["max_abs"] <= 2e-2 * sigma and e["mean_abs"] <= 2e-3 * sigma, (what, e)
    assert e["normwise"] <= NORMWISE["bf16"], (what, e)
    return e


def dev(*xs, dtype):
    return [to_dev(x, dtype) for x in xs]


def synced(o):
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    return from_dev(o)


def push_queries(q, dtype, rows, value=-30.0):
    """q with the given query rows set to `value` (every component)."""
    q = q.copy()
    if dtype == "bf16":
        q[..., rows, :] = workloads.f32_to_bf16_bits(np.full((1,), value, np.float32))[0]
    else:
        q[..., rows, :] = value
    return q


# (dtype, B, H, N, dk, dv, chunk): tensor-core shapes (bf16, dk = dv in {64, 128},
# chunk 128) and CUDA-core shapes (fp32; bf16 with dk != dv or chunk 64).
CAUSAL_SHAPES = [("bf16", 2, 3, 1000, 64, 64, 128), ("bf16", 1, 2, 600, 128, 128, 128),
                 ("bf16", 4, 8, 2048, 64, 64, 128), ("f32", 2, 2, 300, 64, 64, 64),
                 ("f32", 1, 2, 257, 32, 128, 128), ("bf16", 2, 2, 300, 64, 32, 64)]
NONCAUSAL_SHAPES = [("bf16", 2, 3, 1000, 64, 64), ("bf16", 1, 2, 600, 128, 128), ("f32", 2, 2, 300, 64, 32),
                    ("bf16", 2, 2, 300, 128, 64)]


@pytest.mark.parametrize("eps", [1e4, 1e8])
@pytest.mark.parametrize("dtype,B,H,N,dk,dv,chunk", CAUSAL_SHAPES)
def test_causal_clamp_binds(orc, eps, dtype, B, H, N, dk, dv, chunk):
    q, k, v = workloads.random_inputs(31000 + N + dk + dv, B, H, N, dk, dv, dtype)
    o = la().la_forward_causal(*dev(q, k, v, dtype=dtype), chunk=chunk, eps=eps)
    check(synced(o), orc.causal_recurrent(q, k, v, eps), dtype, ("causal clamp", eps, dtype, N, dk, dv, chunk))


@pytest.mark.parametrize("eps", [1e4, 1e8])
@pytest.mark.parametrize("dtype,B,H,N,dk,dv", NONCAUSAL_SHAPES)
def test_noncausal_clamp_binds(orc, eps, dtype, B, H, N, dk, dv):
    q, k, v = workloads.random_inputs(32000 + N + dk + dv, B, H, N, dk, dv, dtype)
    o = la().la_forward_noncausal(*dev(q, k, v, dtype=dtype), eps=eps)
    check(synced(o), orc.noncausal(q, k, v, eps), dtype, ("noncausal clamp", eps, dtype, N, dk, dv))


# Rows whose clamp binds because phi(q) ~ exp(-30): their output is phi(q)^T S / eps,
# so phi(q)'s own relative error reaches it unscaled.  The tensor-core paths evaluate
# exp(x) from x log2(e) rounded to bf16 (relative error <= 2^(|x| log2(e) 2^-9) - 1,
# 9% at x = -30); the CUDA-core paths in fp32.  Their absolute error stays far inside
# the bf16 bounds (|o| ~ 1e-5 there), and on their own scale those rows are held to
# 0.1 (bf16) and 1e-5 (fp32) normwise.
DEAD_ROWS_NORMWISE = {"f32": 1e-5, "bf16": 0.1}


@pytest.mark.parametrize("dtype,B,H,N,dk,dv,chunk", CAUSAL_SHAPES)
def test_causal_dead_queries_clamp_at_default_eps(orc, dtype, B, H, N, dk, dv, chunk):
    """Every 7th query row at -30: phi(q).z ~ 1e-13 * N < 1e-6, so those rows are
    phi(q)^T S / eps; the other rows are unclamped."""
    q, k, v = workloads.random_inputs(33000 + N + dk + dv, B, H, N, dk, dv, dtype)
    rows = np.arange(0, N, 7)
    q = push_queries(q, dtype, rows)
    o = la().la_forward_causal(*dev(q, k, v, dtype=dtype), chunk=chunk)
    got, ref = synced(o), orc.causal_recurrent(q, k, v)
    check(got, ref, dtype, ("dead queries", dtype, N, dk, dv, chunk))
    # the clamped rows on their own scale (they are ~1e-5 of the others)
    e = errors(got[..., rows, :], ref[..., rows, :])
    assert e["normwise"] <= DEAD_ROWS_NORMWISE[dtype], e


@pytest.mark.parametrize("dtype,B,H,N,dk,dv", NONCAUSAL_SHAPES)
def test_noncausal_dead_queries_clamp_at_default_eps(orc, dtype, B, H, N, dk, dv):
    q, k, v = workloads.random_inputs(34000 + N + dk + dv, B, H, N, dk, dv, dtype)
    rows = np.arange(3, N, 11)
    q = push_queries(q, dtype, rows)
    o = la().la_forward_noncausal(*dev(q, k, v, dtype=dtype))
    got, ref = synced(o), orc.noncausal(q, k, v)
    check(got, ref, dtype, ("noncausal dead queries", dtype, N, dk, dv))
    e = errors(got[..., rows, :], ref[..., rows, :])
    assert e["normwise"] <= DEAD_ROWS_NORMWISE[dtype], e


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_decode_clamp_binds(orc, dtype, d):
    """A 30-token prefill, then steps with eps = 1e8, then steps with queries at -30
    and the default eps."""
    B, H, P, T = 2, 5, 30, 6
    q, k, v = workloads.random_inputs(35000 + d, B, H, P + 2 * T, d, d, dtype)
    S, z = la().la_prefill_state(*dev(k[:, :, :P], v[:, :, :P], dtype=dtype))
    Sr, zr = orc.prefill_state(k[:, :, :P], v[:, :, :P])
    for t in range(P, P + 2 * T):
        eps = 1e8 if t < P + T else 1e-6
        qt = q[:, :, t] if t < P + T else push_queries(q[:, :, t:t + 1], dtype, [0])[:, :, 0]
        o = la().la_decode_step(S, z, *dev(qt, k[:, :, t], v[:, :, t], dtype=dtype), eps=eps)
        ref = orc.decode_step(Sr, zr, qt, k[:, :, t], v[:, :, t], eps)
        check(synced(o), ref, dtype, ("decode clamp", dtype, d, t))


@pytest.mark.parametrize("eps", [1e4, 1e8])
@pytest.mark.parametrize("dtype,N,d,chunk", [("bf16", 1000, 64, 128), ("bf16", 700, 128, 128),
                                             ("f32", 300, 64, 64)])
def test_decayed_causal_clamp_binds(orc, eps, dtype, N, d, chunk):
    B, H = 2, 4
    q, k, v = workloads.random_inputs(36000 + N + d, B, H, N, d, d, dtype)
    gamma = workloads.decay_gammas(H)
    g = torch.from_numpy(gamma).cuda()
    o = la().la_forward_causal_decay(*dev(q, k, v, dtype=dtype), g, chunk=chunk, eps=eps)
    ref = orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64), eps)
    check(synced(o), ref, dtype, ("decay clamp", eps, dtype, N, d))


@pytest.mark.parametrize("eps", [1e4, 1e8])
@pytest.mark.parametrize("dtype,N,d", [("bf16", 1000, 64), ("bf16", 600, 128), ("f32", 300, 64)])
def test_variant_clamp_binds(orc, eps, dtype, N, d):
    """ReLU + 0.25 with the normaliser, causal and non-causal."""
    B, H = 2, 3
    q, k, v = workloads.random_inputs(37000 + N + d, B, H, N, d, d, dtype)
    qd, kd, vd = dev(q, k, v, dtype=dtype)
    o = la().la_forward_causal_ex(qd, kd, vd, feature_map="relu", shift=0.25, eps=eps)
    ref = orc.causal_general(q, k, v, fmap="relu", shift=0.25, eps=eps)
    check(synced(o), ref, dtype, ("relu causal clamp", eps, dtype, N, d))
    o = la().la_forward_noncausal_ex(qd, kd, vd, feature_map="relu", shift=0.25, eps=eps)
    ref = orc.noncausal_general(q, k, v, fmap="relu", shift=0.25, eps=eps)
    check(synced(o), ref, dtype, ("relu noncausal clamp", eps, dtype, N, d))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_clamp_binds(orc, dtype):
    """eps = 1e4: the clamp binds on the early rows only; no gradient flows into
    the denominator there.  Gradient errors scaled by the largest reference
    gradient: <= 1e-5 (fp32), <= 1e-2 (bf16).  The decision den > eps is taken in
    each side's own precision; in bf16 (the tensor-core path sums the bf16-rounded
    scores) a row whose float64 denominator lies within 1% of eps may fall on the
    other side, which changes that row's dq by about dd * z: those rows (checked
    to be few) are left out of the dq comparison, dk and dv are compared in full."""
    B, H, N, d = 2, 3, 300, 64
    eps = 1e4
    q, k, v = workloads.random_inputs(38000, B, H, N, d, d, dtype)
    dout = workloads.random_inputs(38001, B, H, N, d, d, dtype)[2]
    got = la().la_backward_causal(*dev(q, k, v, dout, dtype=dtype), eps=eps)
    torch.cuda.synchronize()
    ref = orc.causal_backward(q, k, v, dout, eps)
    scale = max(float(np.max(np.abs(r))) for r in ref)
    tol = 1e-5 if dtype == "f32" else 1e-2
    keep = np.ones((B, H, N), bool)
    if dtype == "bf16":
        phi = lambda x: np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
        fq = phi(workloads.bf16_bits_to_f32(q).astype(np.float64))  # q, k: bf16 bit patterns
        fk = phi(workloads.bf16_bits_to_f32(k).astype(np.float64))
        den = np.einsum("bhnd,bhnd->bhn", fq, np.cumsum(fk, axis=2))
        keep = np.abs(den / eps - 1.0) > 1e-2
        assert keep.mean() > 0.95, float(keep.mean())
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        d_ = np.abs(from_dev(g) - r)
        if name == "dq":
            d_ = d_[keep]
        assert d_.max() <= tol * scale, (name, float(d_.max()), scale)


# ------------------------------------------------------------------ large inputs
@pytest.mark.parametrize("sigma", [2.0, 4.0])
@pytest.mark.parametrize("B,H,N,d", [(4, 8, 2048, 64), (1, 4, 8192, 128), (2, 3, 1000, 64)])
def test_causal_tensor_core_large_inputs(orc, sigma, B, H, N, d):
    """The headline shape (B4 H8 N2048 d64) and a long d = 128 shape at sigma 2 and 4."""
    q, k, v = workloads.random_inputs(39000 + N + d + int(sigma), B, H, N, d, d, "bf16", sigma)
    o = la().la_forward_causal(*dev(q, k, v, dtype="bf16"))
    check_scaled(synced(o), orc.causal_recurrent(q, k, v), sigma, ("causal sigma", sigma, B, H, N, d))


@pytest.mark.parametrize("sigma", [2.0, 4.0])
@pytest.mark.parametrize("B,H,N,d", [(8, 12, 4096, 64), (2, 3, 3000, 128)])
def test_noncausal_tensor_core_large_inputs(orc, sigma, B, H, N, d):
    q, k, v = workloads.random_inputs(40000 + N + d + int(sigma), B, H, N, d, d, "bf16", sigma)
    o = la().la_forward_noncausal(*dev(q, k, v, dtype="bf16"))
    check_scaled(synced(o), orc.noncausal(q, k, v), sigma, ("noncausal sigma", sigma, B, H, N, d))


@pytest.mark.parametrize("sigma", [2.0, 4.0])
def test_decayed_and_prefill_large_inputs(orc, sigma):
    B, H, N, d = 2, 4, 1000, 64
    q, k, v = workloads.random_inputs(41000 + int(sigma), B, H, N, d, d, "bf16", sigma)
    gamma = workloads.decay_gammas(H)
    o = la().la_forward_causal_decay(*dev(q, k, v, dtype="bf16"), torch.from_numpy(gamma).cuda())
    check_scaled(synced(o), orc.causal_decay_recurrent(q, k, v, gamma.astype(np.float64)), sigma,
                 ("decay sigma", sigma))
    S, z = la().la_prefill_state(*dev(k, v, dtype="bf16"))
    torch.cuda.synchronize()
    Sr, zr = orc.prefill_state(k, v)
    assert errors(from_dev(S), Sr)["normwise"] < 1e-5 and errors(from_dev(z), zr)["normwise"] < 1e-5


# ------------------------------------------------------------------ o_0 = v_0
@pytest.mark.parametrize("d,N", [(64, 130), (64, 2048), (128, 300)])
def test_causal_tensor_core_output0_is_v0_exactly(d, N):
    """bf16, chunk 128, dk = dv in {64, 128}: the tensor-core path.  q_0 scaled by
    10 (bf16 rounding of the scaled values is exact or not: any q_0 will do)."""
    q, k, v = workloads.random_inputs(42000 + d + N, 2, 4, N, d, d, "bf16")
    q0 = workloads.bf16_bits_to_f32(q[..., 0, :]) * 10.0
    q[..., 0, :] = workloads.f32_to_bf16_bits(q0.astype(np.float32))
    o = synced(la().la_forward_causal(*dev(q, k, v, dtype="bf16")))
    v0 = workloads.bf16_bits_to_f32(v[..., 0, :]).astype(np.float64)
    assert np.array_equal(o[..., 0, :], v0)


# ------------------------------------------------------------------ identity map, normalised
@pytest.mark.parametrize("dtype,N,d,chunk", [("bf16", 1000, 64, 128), ("bf16", 600, 128, 128),
                                             ("f32", 300, 64, 64)])
def test_identity_map_normalised_where_defined(orc, dtype, N, d, chunk):
    """phi(x) = x + 8 on N(0, 1) inputs is positive (x > -8), so the normalised form
    is a convex combination of the v_j like elu + 1: causal, non-causal and decode."""
    B, H = 2, 3
    q, k, v = workloads.random_inputs(43000 + N + d, B, H, N, d, d, dtype)
    assert workloads.bf16_bits_to_f32(q).min() > -8 if dtype == "bf16" else q.min() > -8
    qd, kd, vd = dev(q, k, v, dtype=dtype)
    o = la().la_forward_causal_ex(qd, kd, vd, feature_map="identity", shift=8.0, normalize=True, chunk=chunk)
    ref = orc.causal_general(q, k, v, fmap="identity", shift=8.0, normalize=True)
    check(synced(o), ref, dtype, ("identity causal", dtype, N, d))
    o = la().la_forward_noncausal_ex(qd, kd, vd, feature_map="identity", shift=8.0, normalize=True)
    ref = orc.noncausal_general(q, k, v, fmap="identity", shift=8.0, normalize=True)
    check(synced(o), ref, dtype, ("identity noncausal", dtype, N, d))
    S, z = la().la_prefill_state_ex(kd, vd, feature_map="identity", shift=8.0)
    Sr, zr = orc.prefill_state_general(k, v, fmap="identity", shift=8.0)
    for t in range(3):
        qt, kt, vt = workloads.random_inputs(43100 + t, B, H, 1, d, d, dtype)
        o = la().la_decode_step_ex(S, z, *dev(qt[:, :, 0], kt[:, :, 0], vt[:, :, 0], dtype=dtype),
                                   feature_map="identity", shift=8.0, normalize=True)
        ref = orc.decode_step_general(Sr, zr, qt[:, :, 0], kt[:, :, 0], vt[:, :, 0], fmap="identity", shift=8.0,
                                      normalize=True)
        check(synced(o), ref, dtype, ("identity decode", dtype, d, t))


# ------------------------------------------------------------------ guard canaries
PAD = 256


def padded(shape, dtype):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * PAD,), 12345.0, dtype=dtype, device="cuda")
    return buf, buf[PAD:PAD + n].view(shape)


def untouched(buf):
    return bool(torch.all(buf[:PAD] == 12345.0)) and bool(torch.all(buf[-PAD:] == 12345.0))


@pytest.mark.parametrize("path", ["causal_favor", "noncausal_favor", "favor_features", "backward", "causal_decay",
                                  "decode_decay", "causal_variant", "noncausal_variant", "prefill_state"])
def test_more_output_guard_canaries(path):
    """Every output written into the middle of a sentinel-filled buffer: the padding
    on both sides stays untouched and the output is finite."""
    B, H, N, d = 2, 3, 150, 64
    dt = torch.bfloat16
    gen = torch.Generator(device="cuda").manual_seed(6)
    x = torch.randn((B, H, N, d), device="cuda", generator=gen).to(dt)
    w = (0.5 * torch.randn((d, d), device="cuda", generator=gen)).to(dt)
    gamma = torch.full((H,), 0.9, device="cuda")
    bufs = []
    if path in ("causal_favor", "noncausal_favor"):
        b, o = padded(x.shape, dt)
        bufs.append((b, o))
        if path == "causal_favor":
            la().la_forward_causal_favor(x, x, x, w, o=o)
        else:
            la().la_forward_noncausal_favor(x, x, x, w, o=o)
    elif path == "favor_features":
        b, o = padded(x.shape, dt)
        bufs.append((b, o))
        la().la_favor_features(x, w, phi=o)
    elif path == "backward":
        outs = [padded(x.shape, dt) for _ in range(3)]
        bufs += outs
        la().la_backward_causal(x, x, x, x, dq=outs[0][1], dk=outs[1][1], dv=outs[2][1])
    elif path == "causal_decay":
        b, o = padded(x.shape, dt)
        bufs.append((b, o))
        la().la_forward_causal_decay(x, x, x, gamma, o=o)
    elif path == "decode_decay":
        b, o = padded((B, H, d), dt)
        bufs.append((b, o))
        S = torch.zeros((B, H, d, d), device="cuda")
        z = torch.zeros((B, H, d), device="cuda")
        la().la_decode_step_decay(S, z, *(x[:, :, i].contiguous() for i in range(3)), gamma, o=o)
    elif path == "causal_variant":
        b, o = padded(x.shape, dt)
        bufs.append((b, o))
        la().la_forward_causal_ex(x, x, x, o=o, feature_map="relu", shift=0.1, normalize=False)
    elif path == "noncausal_variant":
        b, o = padded(x.shape, dt)
        bufs.append((b, o))
        la().la_forward_noncausal_ex(x, x, x, o=o, feature_map="relu", shift=0.1, normalize=False)
    else:
        bS, S = padded((B, H, d, d), torch.float32)
        bz, z = padded((B, H, d), torch.float32)
        bufs += [(bS, S), (bz, z)]
        la().la_prefill_state(x, x, S, z)
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    for b, o in bufs:
        assert untouched(b), path
        assert bool(torch.isfinite(o.float()).all()), path



# ------------------------------------------------------------------ per-thread default streams
def test_per_thread_default_streams_get_their_own_workspaces(orc):
    """Two host threads, one after the other, call the bf16 tensor-core forwards on
    cudaStreamPerThread (each thread's own stream, whose workspaces are keyed by the
    thread as well as the handle) while the main thread's work on another stream is
    still queued: every result matches the oracle.  The threads make no CUDA call of
    their own before the library's (it binds the primary context to a thread that
    has none)."""
    import ctypes
    import threading
    lib = la().load_library()
    per_thread = ctypes.c_void_p(2)  # cudaStreamPerThread
    cases = [workloads.random_inputs(44000 + t, 4, 8, 4096, 64, 64, "bf16") for t in range(2)]
    refs = [(orc.causal_recurrent(*c), orc.noncausal(*c)) for c in cases]
    devs = [dev(*c, dtype="bf16") for c in cases]
    reps = 3
    outs = [[[torch.empty_like(d[2]) for _ in range(2)] for _ in range(reps)] for d in devs]
    torch.cuda.synchronize()
    status = [[], []]

    def worker(t):
        q, k, v = devs[t]
        B, H, N, d = q.shape
        for r in range(reps):
            status[t].append(lib.la_forward_causal(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                   outs[t][r][0].data_ptr(), B, H, N, d, d, 128, ctypes.c_float(1e-6),
                                                   1, per_thread))
            status[t].append(lib.la_forward_noncausal(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                      outs[t][r][1].data_ptr(), B, H, N, d, d, ctypes.c_float(1e-6),
                                                      1, per_thread))
        status[t].append(int(torch.cuda.synchronize() is None))

    for t in range(2):  # one thread after the other
        th = threading.Thread(target=worker, args=(t,))
        th.start()
        th.join(timeout=120)
        assert not th.is_alive()
    torch.cuda.synchronize()
    assert la().la_get_device_status() == 0
    for t in range(2):
        assert all(st == 0 for st in status[t][:-1]), status[t]
        for r in range(reps):
            check(from_dev(outs[t][r][0]), refs[t][0], "bf16", ("per-thread causal", t, r))
            check(from_dev(outs[t][r][1]), refs[t][1], "bf16", ("per-thread noncausal", t, r))
