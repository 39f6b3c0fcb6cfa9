"""Pins for the float64 oracle: checks against facts the pages and mathematics fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a violation.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on builds with a planted mistake and
requires that every such build fails at least one pin.

None of these re-types the oracle's own loop: the references are exact
rational arithmetic (fractions), a brute-force pairwise form written here with
numpy, library routines (math.expm1), or identities the method must satisfy.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import workloads

EPS = 1e-6


# ----------------------------------------------------------------------------
# references written independently of the oracle
# ----------------------------------------------------------------------------
def elu_plus_one_ref(x: float) -> float:
    """elu(x) + 1 with alpha = 1 via the library's expm1 (elu(x) = expm1(x) for x <= 0)."""
    return (x if x > 0 else math.expm1(x)) + 1.0


def phi_np(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def pairwise_bruteforce(q, k, v, causal: bool, eps: float = EPS) -> np.ndarray:
    """Similarity-weighted average, general form sum_j sim(q_i,k_j) v_j / sum_j sim(q_i,k_j)
    ("Linear attention", learn.pranaymahendrakar.com, Researcher: Derivation), with
    sim = phi(q).phi(k); for causal, j <= i.  Dense N x N numpy, float64."""
    fq, fk = phi_np(q), phi_np(k)
    v = np.asarray(v, dtype=np.float64)
    scores = fq @ np.swapaxes(fk, -1, -2)
    if causal:
        n = scores.shape[-1]
        scores = scores * np.tril(np.ones((n, n)))
    den = np.maximum(scores.sum(-1, keepdims=True), eps)
    return (scores @ v) / den


def exact_causal(qf, kf, v, causal=True):
    """Exact rational o for inputs whose phi values are given as Fractions.

    qf, kf: lists [N][d] of Fraction (already phi-mapped), v: [N][dv] Fraction.
    """
    N, dv = len(qf), len(v[0])
    out = []
    for i in range(N):
        js = range(i + 1) if causal else range(N)
        num = [Fraction(0)] * dv
        den = Fraction(0)
        for j in js:
            s = sum(a * b for a, b in zip(qf[i], kf[j]))
            den += s
            for c in range(dv):
                num[c] += s * v[j][c]
        out.append([x / den for x in num])
    return out


def _rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _rand(seed, BH, N, dk, dv, sigma=1.0):
    q, k, v = workloads.random_inputs(seed, 1, BH, N, dk, dv, "f32", sigma)
    return q[0].astype(np.float64), k[0].astype(np.float64), v[0].astype(np.float64)


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------
def pin_phi_is_elu_plus_one(orc):
    """phi = elu + 1 (alpha 1): matches expm1-based elu, is continuous at 0 and > 0."""
    xs = [-50.0, -20.0, -3.5, -1.0, -0.25, -1e-9, 0.0, 1e-9, 0.3, 1.0, 2.5, 40.0]
    for x in xs:
        got, ref = orc.phi(x), elu_plus_one_ref(x)
        assert abs(got - ref) <= 1e-15 * max(1.0, abs(ref)), (x, got, ref)
        assert got > 0.0
    assert orc.phi(0.0) == 1.0


def pin_output0_equals_v0(orc):
    """Position 0 returns v_0 for any q_0 ("26. Linear (Kernelized) Attention",
    Step-by-Step step 6), as long as the denominator is above eps."""
    rng = np.random.default_rng(123)
    for scale in (1.0, 10.0, 30.0):
        for dk, dv in ((3, 2), (8, 5), (32, 32)):
            q = rng.standard_normal((2, 4, dk)) * scale
            k = rng.standard_normal((2, 4, dk))
            v = rng.standard_normal((2, 4, dv))
            for o in (orc.causal_recurrent(q, k, v, EPS), orc.causal_chunked(q, k, v, 2, EPS),
                      orc.causal_quadratic(q, k, v, EPS)):
                den = (phi_np(q[:, 0]) * phi_np(k[:, 0])).sum(-1)
                ok = den > EPS
                assert np.all(np.abs(o[ok, 0] - v[ok, 0]) <= 1e-14 * (1 + np.abs(v[ok, 0]))), scale


def pin_eps_clamp(orc):
    """Below eps the denominator is clamped: o_0 = v_0 * den / eps (the clamp of the
    chunked listing of "Linear Attention", aiwiki.thehackersbrain.dev)."""
    q = np.full((1, 1, 4), -12.0)
    k = np.full((1, 1, 4), -12.0)
    v = np.array([[[0.5, -2.0, 3.0]]])
    den = 4 * math.exp(-12.0) * math.exp(-12.0)   # ~1.5e-10 < eps
    assert den < EPS
    for o in (orc.causal_recurrent(q, k, v, EPS), orc.noncausal(q, k, v, EPS),
              orc.causal_chunked(q, k, v, 1, EPS)):
        ref = v[0, 0] * (den / EPS)
        assert np.allclose(o[0, 0], ref, rtol=1e-12, atol=0), (o, ref)


def pin_exact_rational(orc):
    """Tiny inputs with q, k > 0 (phi = x + 1 is exact) against exact rational
    arithmetic of the similarity-weighted form; dk != dv so a transposed or
    mis-indexed operand changes the answer."""
    rng = np.random.default_rng(5)
    N, dk, dv = 7, 3, 4
    qd = rng.integers(1, 9, size=(N, dk)) / 4.0     # positive dyadic values
    kd = rng.integers(1, 9, size=(N, dk)) / 8.0
    vd = rng.integers(-6, 7, size=(N, dv)) / 2.0
    qf = [[Fraction(x) + 1 for x in row] for row in qd]
    kf = [[Fraction(x) + 1 for x in row] for row in kd]
    vf = [[Fraction(x) for x in row] for row in vd]
    for causal in (True, False):
        ref = np.array([[float(x) for x in row] for row in exact_causal(qf, kf, vf, causal)])
        if causal:
            outs = [orc.causal_recurrent(qd, kd, vd, EPS), orc.causal_quadratic(qd, kd, vd, EPS)]
            outs += [orc.causal_chunked(qd, kd, vd, c, EPS) for c in (1, 2, 3, 7, 9)]
        else:
            outs = [orc.noncausal(qd, kd, vd, EPS), orc.noncausal_pairwise(qd, kd, vd, EPS)]
        for o in outs:
            assert np.allclose(o, ref, rtol=1e-14, atol=1e-14), (causal, np.max(np.abs(o - ref)))


def pin_exact_rational_state(orc):
    """Prefill state S = sum phi(k) v^T, z = sum phi(k) in exact arithmetic."""
    rng = np.random.default_rng(6)
    N, dk, dv = 5, 4, 3
    kd = rng.integers(1, 9, size=(2, N, dk)) / 4.0
    vd = rng.integers(-5, 6, size=(2, N, dv)) / 4.0
    S, z = orc.prefill_state(kd, vd)
    for b in range(2):
        for r in range(dk):
            zr = sum(Fraction(kd[b, t, r]) + 1 for t in range(N))
            assert float(zr) == z[b, r]
            for c in range(dv):
                s = sum((Fraction(kd[b, t, r]) + 1) * Fraction(vd[b, t, c]) for t in range(N))
                assert float(s) == S[b, r, c], (b, r, c)


def pin_noncausal_equals_pairwise(orc):
    """Non-causal associative form equals the brute-force pairwise form
    ("Linear attention: change the order.", implementation you can check), both
    against the numpy brute force here and the oracle's own pairwise form."""
    for seed, (N, dk, dv) in enumerate(((1, 1, 1), (5, 3, 1), (17, 8, 3), (64, 3, 8), (33, 8, 8))):
        q, k, v = _rand(100 + seed, 3, N, dk, dv)
        ref = pairwise_bruteforce(q, k, v, causal=False)
        assert _rel_err(orc.noncausal(q, k, v, EPS), ref) < 1e-12
        assert _rel_err(orc.noncausal_pairwise(q, k, v, EPS), ref) < 1e-12


def pin_causal_equals_masked_bruteforce(orc):
    """Causal recurrence equals the masked quadratic form ("Linear attention",
    Developer listing, part 3: the load-bearing check) on tiny inputs."""
    for seed, (N, dk, dv) in enumerate(((1, 1, 1), (9, 3, 2), (40, 8, 3), (64, 5, 8))):
        q, k, v = _rand(200 + seed, 2, N, dk, dv)
        ref = pairwise_bruteforce(q, k, v, causal=True)
        assert _rel_err(orc.causal_recurrent(q, k, v, EPS), ref) < 1e-12
        assert _rel_err(orc.causal_quadratic(q, k, v, EPS), ref) < 1e-12


def pin_chunked_equals_recurrent_every_chunk(orc):
    """Chunked form equals the recurrence for every chunk size 1..N and beyond,
    including non-divisors of N ("Linear Attention", chunked listing)."""
    N = 37
    q, k, v = _rand(300, 2, N, 6, 4)
    ref = orc.causal_recurrent(q, k, v, EPS)
    bf = pairwise_bruteforce(q, k, v, causal=True)
    assert _rel_err(ref, bf) < 1e-12
    for c in list(range(1, N + 1)) + [N + 5, 128]:
        assert _rel_err(orc.causal_chunked(q, k, v, c, EPS), ref) < 1e-12, c


def pin_convex_hull(orc):
    """Non-negative weights: every o_i lies within [min_{j<=i} v_j, max_{j<=i} v_j]
    per component ("Linear Attention": a weighted average with non-negative weights)."""
    q, k, v = _rand(400, 3, 200, 8, 6, sigma=2.0)
    o = orc.causal_recurrent(q, k, v, EPS)
    lo = np.minimum.accumulate(v, axis=1)
    hi = np.maximum.accumulate(v, axis=1)
    tol = 1e-12 * (1 + np.abs(v).max())
    assert np.all(o >= lo - tol) and np.all(o <= hi + tol)
    on = orc.noncausal(q, k, v, EPS)
    assert np.all(on >= v.min(axis=1, keepdims=True) - tol)
    assert np.all(on <= v.max(axis=1, keepdims=True) + tol)


def pin_constant_v(orc):
    """Constant v = c gives o = c everywhere (weights sum to the denominator)."""
    q, k, _ = _rand(500, 2, 50, 7, 3)
    v = np.full((2, 50, 3), -1.75)
    for o in (orc.causal_recurrent(q, k, v, EPS), orc.noncausal(q, k, v, EPS),
              orc.causal_chunked(q, k, v, 16, EPS)):
        assert np.allclose(o, -1.75, rtol=1e-13, atol=0)


def pin_linear_in_v(orc):
    """o is linear in v for fixed q, k."""
    q, k, v1 = _rand(600, 2, 30, 5, 4)
    _, _, v2 = _rand(601, 2, 30, 5, 4)
    a, b = 0.75, -2.5
    for f in (orc.causal_recurrent, orc.noncausal):
        lhs = f(q, k, a * v1 + b * v2, EPS)
        rhs = a * f(q, k, v1, EPS) + b * f(q, k, v2, EPS)
        assert _rel_err(lhs, rhs) < 1e-12


def pin_noncausal_permutation_invariant(orc):
    """Non-causal o does not depend on the order of the (k, v) pairs."""
    q, k, v = _rand(700, 2, 45, 6, 5)
    perm = np.random.default_rng(7).permutation(45)
    assert _rel_err(orc.noncausal(q, k[:, perm], v[:, perm], EPS), orc.noncausal(q, k, v, EPS)) < 1e-13


def pin_last_causal_row_is_noncausal(orc):
    """The last causal row sees every key, so it equals the non-causal row."""
    q, k, v = _rand(800, 3, 60, 8, 4)
    oc = orc.causal_recurrent(q, k, v, EPS)
    on = orc.noncausal(q, k, v, EPS)
    assert _rel_err(oc[:, -1], on[:, -1]) < 1e-13
    # and the causal output depends on the sequence order (it is not the non-causal one)
    assert _rel_err(oc[:, 0], on[:, 0]) > 1e-3


def pin_decode_continues_causal(orc):
    """Prefill state of the first P tokens, then single-token decode steps,
    reproduces the causal forward of the whole sequence ("Linear Attention
    -- Math + Variants": parallel form for training, recurrence for decoding)."""
    BH, N, P, dk, dv = 3, 24, 10, 6, 5
    q, k, v = _rand(900, BH, N, dk, dv)
    full = orc.causal_recurrent(q, k, v, EPS)
    S, z = orc.prefill_state(k[:, :P], v[:, :P])
    for t in range(P, N):
        o = orc.decode_step(S, z, q[:, t], k[:, t], v[:, t], EPS)
        assert _rel_err(o, full[:, t]) < 1e-12, t
    # after all steps the state is the prefill state of the whole sequence
    S2, z2 = orc.prefill_state(k, v)
    assert _rel_err(S, S2) < 1e-13 and _rel_err(z, z2) < 1e-13


def pin_bf16_widening(orc):
    """bf16 inputs are widened exactly: the oracle on bf16 bits equals the oracle
    on the float64 values those bits denote."""
    q, k, v = workloads.random_inputs(11, 1, 2, 20, 4, 3, "bf16")
    qf, kf, vf = (workloads.bf16_bits_to_f32(x).astype(np.float64) for x in (q, k, v))
    a = orc.causal_recurrent(q, k, v, EPS)
    b = orc.causal_recurrent(qf, kf, vf, EPS)
    assert np.array_equal(a, b)
    ref = pairwise_bruteforce(qf[0], kf[0], vf[0], causal=True)
    assert _rel_err(a[0], ref) < 1e-12


# ----------------------------------------------------------------------------
# decayed state: S_t = g S_{t-1} + phi(k_t) v_t^T, z likewise ("Linear Attention --
# Math + Variants", RetNet and gated linear attention: a fixed per-head decay;
# "Linear attention", learn.pranaymahendrakar.com, Try it yourself)
# ----------------------------------------------------------------------------
def weighted_pairwise(q, k, v, g, eps=EPS):
    """sum_{j<=i} g^(i-j) phi(q_i).phi(k_j) v_j / sum_{j<=i} g^(i-j) phi(q_i).phi(k_j),
    dense numpy per sequence (leading dim = sequences, g one value per sequence)."""
    out = []
    for s in range(q.shape[0]):
        fq, fk = phi_np(q[s]), phi_np(k[s])
        n = fq.shape[0]
        i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        w = np.where(j <= i, float(g[s]) ** np.maximum(i - j, 0), 0.0)
        scores = (fq @ fk.T) * w
        den = np.maximum(scores.sum(-1, keepdims=True), eps)
        out.append((scores @ np.asarray(v[s], dtype=np.float64)) / den)
    return np.stack(out)


def pin_decay_equals_weighted_pairwise(orc):
    """The decayed recurrence (and the oracle's own weighted quadratic form) equals the
    weighted pairwise form written above, for decays 1, 0.9, 0.5 and 0."""
    q, k, v = _rand(1000, 4, 50, 6, 5)
    g = np.array([1.0, 0.9, 0.5, 0.0])
    ref = weighted_pairwise(q, k, v, g)
    assert _rel_err(orc.causal_decay_recurrent(q, k, v, g, EPS), ref) < 1e-12
    assert _rel_err(orc.causal_decay_quadratic(q, k, v, g, EPS), ref) < 1e-12


def pin_decay_one_is_undecayed(orc):
    """gamma = 1 gives the undecayed causal form, for every head."""
    q, k, v = _rand(1010, 3, 40, 5, 7)
    assert _rel_err(orc.causal_decay_recurrent(q, k, v, np.ones(3), EPS), orc.causal_recurrent(q, k, v, EPS)) < 1e-13


def pin_decay_zero_returns_v(orc):
    """gamma = 0 keeps only the current token: o_t = v_t (phi > 0, so the weight is
    positive and cancels)."""
    q, k, v = _rand(1020, 2, 30, 4, 3)
    assert _rel_err(orc.causal_decay_recurrent(q, k, v, np.zeros(2), EPS), v) < 1e-14


def pin_decay_exact_rational(orc):
    """Tiny inputs with q, k > 0 (phi = x + 1 exact) and gamma = 1/2, against exact
    rational arithmetic of the weighted form."""
    rng = np.random.default_rng(1030)
    N, dk, dv = 6, 3, 2
    qv = rng.integers(1, 8, size=(N, dk)) / 8.0
    kv = rng.integers(1, 8, size=(N, dk)) / 8.0
    vv = rng.integers(-8, 9, size=(N, dv)) / 4.0
    got = orc.causal_decay_recurrent(qv[None], kv[None], vv[None], [0.5], 0.0)[0]
    fq = [[Fraction(x).limit_denominator(64) + 1 for x in row] for row in qv]
    fk = [[Fraction(x).limit_denominator(64) + 1 for x in row] for row in kv]
    vf = [[Fraction(x).limit_denominator(64) for x in row] for row in vv]
    for i in range(N):
        num = [Fraction(0)] * dv
        den = Fraction(0)
        for j in range(i + 1):
            s = sum(a * b for a, b in zip(fq[i], fk[j])) * Fraction(1, 2) ** (i - j)
            den += s
            for c in range(dv):
                num[c] += s * vf[j][c]
        for c in range(dv):
            assert abs(got[i, c] - float(num[c] / den)) <= 1e-14 * max(1.0, abs(float(num[c] / den)))


def pin_decay_differs_from_unweighted(orc):
    """With decay the causal output no longer matches the unweighted quadratic form
    ("Linear attention", Try it yourself), except at the first position."""
    q, k, v = _rand(1040, 2, 30, 4, 3)
    dec = orc.causal_decay_recurrent(q, k, v, np.full(2, 0.9), EPS)
    plain = pairwise_bruteforce(q, k, v, causal=True)
    assert _rel_err(dec[:, 0], plain[:, 0]) < 1e-13
    assert _rel_err(dec[:, 1:], plain[:, 1:]) > 1e-2


def pin_decode_decay_continues_causal(orc):
    """Decayed decode steps from a zero state reproduce the decayed causal forward at
    every position (the step is the recurrence's body)."""
    BH, N, dk, dv = 3, 20, 5, 4
    q, k, v = _rand(1050, BH, N, dk, dv)
    g = np.array([0.95, 0.7, 1.0])
    full = orc.causal_decay_recurrent(q, k, v, g, EPS)
    S = np.zeros((BH, dk, dv))
    z = np.zeros((BH, dk))
    for t in range(N):
        o = orc.decode_step_decay(S, z, q[:, t], k[:, t], v[:, t], g, EPS)
        assert _rel_err(o, full[:, t]) < 1e-12, t
    assert _rel_err(o, weighted_pairwise(q, k, v, g)[:, -1]) < 1e-12


# ----------------------------------------------------------------------------
# feature maps and the normaliser ("Linear attention", What the pieces are for:
# ReLU; "Linear Attention -- Math + Variants", Feature-map families: ReLU and
# identity-plus-shift, Implementation reality: dropping the normaliser;
# "26. Linear (Kernelized) Attention", Key Functions & Tricks: relu(x) + eps)
# ----------------------------------------------------------------------------
def feature_np(x, fmap, shift):
    x = np.asarray(x, dtype=np.float64)
    if fmap == "relu":
        return np.maximum(x, 0.0) + shift
    if fmap == "identity":
        return x + shift
    return phi_np(x)


def general_pairwise(q, k, v, g, fmap, shift, normalize, causal=True, eps=EPS):
    """Dense numpy per sequence: scores g^(i-j) f(q_i).f(k_j) (j <= i when causal;
    g = None: no decay), o = scores v, divided by max(row sums, eps) when normalize."""
    out = []
    for s in range(q.shape[0]):
        fq, fk = feature_np(q[s], fmap, shift), feature_np(k[s], fmap, shift)
        n = fq.shape[0]
        i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        w = np.ones((n, n)) if g is None else float(g[s]) ** np.maximum(i - j, 0)
        if causal:
            w = np.where(j <= i, w, 0.0)
        scores = (fq @ fk.T) * w
        o = scores @ np.asarray(v[s], dtype=np.float64)
        if normalize:
            o = o / np.maximum(scores.sum(-1, keepdims=True), eps)
        out.append(o)
    return np.stack(out)


def pin_general_default_is_the_pinned_forms(orc):
    """The general recurrence with elu + 1 and the normaliser is the pinned causal
    form, with a decay the pinned decayed form (bit for bit: same arithmetic)."""
    q, k, v = _rand(2000, 3, 25, 5, 4)
    assert np.array_equal(orc.causal_general(q, k, v), orc.causal_recurrent(q, k, v, EPS))
    g = np.array([0.9, 0.5, 1.0])
    assert np.array_equal(orc.causal_general(q, k, v, gamma=g), orc.causal_decay_recurrent(q, k, v, g, EPS))


def pin_general_equals_numpy_pairwise(orc):
    """Every map x normaliser x decay against the dense numpy form above (and the
    oracle's own quadratic form against it too)."""
    q, k, v = _rand(2010, 3, 40, 6, 5)
    for fmap, shift in (("relu", 0.0), ("relu", 0.25), ("identity", 0.5), ("elu1", 0.0)):
        for normalize in (True, False):
            for g in (None, np.array([0.9, 0.6, 1.0])):
                ref = general_pairwise(q, k, v, g, fmap, shift, normalize)
                got = orc.causal_general(q, k, v, gamma=g, fmap=fmap, shift=shift, normalize=normalize)
                assert _rel_err(got, ref) < 1e-12, (fmap, shift, normalize, g is None)
                got = orc.causal_general_quadratic(q, k, v, gamma=g, fmap=fmap, shift=shift, normalize=normalize)
                assert _rel_err(got, ref) < 1e-12, (fmap, shift, normalize, g is None)


def pin_general_exact_integers(orc):
    """Identity map without shift, no normaliser, small integers: every value is an
    integer below 2^53, so the float64 result equals exact integer arithmetic."""
    rng = np.random.default_rng(2020)
    N, dk, dv = 9, 4, 3
    q = rng.integers(-5, 6, size=(1, N, dk)).astype(np.float64)
    k = rng.integers(-5, 6, size=(1, N, dk)).astype(np.float64)
    v = rng.integers(-7, 8, size=(1, N, dv)).astype(np.float64)
    got = orc.causal_general(q, k, v, fmap="identity", shift=0.0, normalize=False)[0]
    qi, ki, vi = q[0].astype(int).tolist(), k[0].astype(int).tolist(), v[0].astype(int).tolist()
    for i in range(N):
        for c in range(dv):
            exact = sum(sum(a * b for a, b in zip(qi[i], ki[j])) * vi[j][c] for j in range(i + 1))
            assert got[i, c] == exact
    # relu + 1 of integers: max(x, 0) + 1, again all integers
    got = orc.causal_general(q, k, v, fmap="relu", shift=1.0, normalize=False)[0]
    fq = [[max(a, 0) + 1 for a in row] for row in qi]
    fk = [[max(a, 0) + 1 for a in row] for row in ki]
    for i in range(N):
        for c in range(dv):
            exact = sum(sum(a * b for a, b in zip(fq[i], fk[j])) * vi[j][c] for j in range(i + 1))
            assert got[i, c] == exact


def pin_unnormalized_ones_is_the_denominator(orc):
    """Without the normaliser, v = 1 gives the denominator sum_j w_ij f(q_i).f(k_j); the
    normalised output is the unnormalised one divided by max(that, eps)."""
    q, k, v = _rand(2030, 2, 30, 5, 4)
    g = np.array([0.8, 1.0])
    ones = np.ones((2, 30, 1))
    for fmap, shift in (("relu", 0.1), ("elu1", 0.0), ("identity", 3.0)):
        den = orc.causal_general(q, k, ones, gamma=g, fmap=fmap, shift=shift, normalize=False)
        raw = orc.causal_general(q, k, v, gamma=g, fmap=fmap, shift=shift, normalize=False)
        nrm = orc.causal_general(q, k, v, gamma=g, fmap=fmap, shift=shift, normalize=True)
        assert _rel_err(nrm, raw / np.maximum(den, EPS)) < 1e-13, fmap


def pin_relu_dead_queries_give_zero(orc):
    """ReLU without shift: a query with no positive component has f(q) = 0, so the
    numerator is 0 and the clamped denominator eps gives o = 0 (normalised or not)."""
    q, k, v = _rand(2040, 2, 20, 4, 3)
    q = -np.abs(q)
    for normalize in (True, False):
        o = orc.causal_general(q, k, v, fmap="relu", shift=0.0, normalize=normalize)
        assert np.all(o == 0.0)


def pin_relu_on_nonnegative_is_identity(orc):
    """For q, k >= 0, max(x, 0) + c = x + c: the two maps agree exactly."""
    q, k, v = _rand(2050, 2, 20, 4, 3)
    q, k = np.abs(q), np.abs(k)
    for normalize in (True, False):
        a = orc.causal_general(q, k, v, fmap="relu", shift=0.3, normalize=normalize)
        b = orc.causal_general(q, k, v, fmap="identity", shift=0.3, normalize=normalize)
        assert np.array_equal(a, b)


def pin_general_noncausal_equals_pairwise(orc):
    q, k, v = _rand(2060, 3, 30, 5, 4)
    for fmap, shift in (("relu", 0.0), ("relu", 0.5), ("identity", 2.0), ("elu1", 0.0)):
        for normalize in (True, False):
            ref = general_pairwise(q, k, v, None, fmap, shift, normalize, causal=False)
            got = orc.noncausal_general(q, k, v, fmap=fmap, shift=shift, normalize=normalize)
            assert _rel_err(got, ref) < 1e-12, (fmap, normalize)


def pin_general_prefill_state(orc):
    """S = sum_t g^(N-1-t) f(k_t) v_t^T, z = sum_t g^(N-1-t) f(k_t), as numpy sums."""
    BH, N, dk, dv = 3, 25, 5, 4
    q, k, v = _rand(2070, BH, N, dk, dv)
    g = np.array([0.9, 0.0, 1.0])
    for fmap, shift in (("relu", 0.2), ("identity", 0.0), ("elu1", 0.0)):
        S, z = orc.prefill_state_general(k, v, gamma=g, fmap=fmap, shift=shift)
        fk = feature_np(k, fmap, shift)
        w = g[:, None] ** (N - 1 - np.arange(N))[None, :]
        Sr = np.einsum("bt,btr,btc->brc", w, fk, v)
        zr = np.einsum("bt,btr->br", w, fk)
        assert _rel_err(S, Sr) < 1e-12 and _rel_err(z, zr) < 1e-12, fmap


def pin_general_decode_continues_causal(orc):
    """General decode steps from a zero state reproduce the general causal forward."""
    BH, N, dk, dv = 3, 16, 5, 4
    q, k, v = _rand(2080, BH, N, dk, dv)
    g = np.array([0.95, 0.5, 1.0])
    for fmap, shift, normalize in (("relu", 0.1, True), ("identity", 0.0, False), ("relu", 0.0, False)):
        full = orc.causal_general(q, k, v, gamma=g, fmap=fmap, shift=shift, normalize=normalize)
        S = np.zeros((BH, dk, dv))
        z = np.zeros((BH, dk))
        for t in range(N):
            o = orc.decode_step_general(S, z, q[:, t], k[:, t], v[:, t], gamma=g, fmap=fmap, shift=shift,
                                        normalize=normalize)
            assert _rel_err(o, full[:, t]) < 1e-12, (fmap, t)


# ----------------------------------------------------------------------------
# backward pass of the causal form: gradients of L = sum(dO * o).  The pages give
# none; the oracle's chain-rule scans are pinned to finite differences of the
# (already pinned) forward oracle and to closed forms.
# ----------------------------------------------------------------------------
def _finite_difference(orc, q, k, v, dout, h=1e-6):
    def loss(qq, kk, vv):
        return float(np.sum(orc.causal_recurrent(qq, kk, vv, EPS) * dout))
    grads = []
    for which in range(3):
        xs = [q, k, v]
        x = xs[which]
        gx = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = list(xs); args_p[which] = xp
            args_m = list(xs); args_m[which] = xm
            gx[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        grads.append(gx)
    return grads


def pin_backward_equals_finite_differences(orc):
    """Central differences of the forward oracle (h = 1e-6, float64) within 1e-7."""
    rng = np.random.default_rng(3000)
    BH, N, dk, dv = 2, 9, 4, 3
    q, k, v, dout = (rng.standard_normal((BH, N, d)) for d in (dk, dk, dv, dv))
    for got, ref in zip(orc.causal_backward(q, k, v, dout), _finite_difference(orc, q, k, v, dout)):
        assert _rel_err(got, ref) < 1e-7


def pin_backward_dv_dense_form(orc):
    """dv_j = sum_{i>=j} s_ij dO_i / d_i with s = phi(Q) phi(K)^T (dense numpy)."""
    q, k, v = _rand(3010, 3, 30, 5, 4)
    dout = _rand(3011, 3, 30, 5, 4)[2]
    _, _, gv = orc.causal_backward(q, k, v, dout)
    for s_ in range(3):
        fq, fk = phi_np(q[s_]), phi_np(k[s_])
        sc = np.tril(fq @ fk.T)
        d = np.maximum(sc.sum(-1), EPS)
        ref = sc.T @ (dout[s_] / d[:, None])
        assert _rel_err(gv[s_], ref) < 1e-12


def pin_backward_first_output_only(orc):
    """o_0 = v_0 whatever q, k: a loss on position 0 alone gives dq = dk = 0 and
    dv = dO at position 0 only."""
    q, k, v = _rand(3020, 2, 12, 4, 3)
    dout = np.zeros_like(v)
    dout[:, 0] = _rand(3021, 2, 1, 4, 3)[2][:, 0]
    gq, gk, gv = orc.causal_backward(q, k, v, dout)
    assert np.max(np.abs(gq)) < 1e-14 and np.max(np.abs(gk)) < 1e-14
    assert _rel_err(gv[:, 0], dout[:, 0]) < 1e-14 and np.max(np.abs(gv[:, 1:])) < 1e-14


def pin_backward_constant_v(orc):
    """With every v_j equal, o_i = v for all i: no gradient reaches q or k, and dv
    sums to sum_i dO_i (the weights of each row sum to one)."""
    q, k, _ = _rand(3030, 2, 20, 5, 3)
    v = np.broadcast_to(np.array([0.5, -1.0, 2.0]), (2, 20, 3)).copy()
    dout = _rand(3031, 2, 20, 5, 3)[2]
    gq, gk, gv = orc.causal_backward(q, k, v, dout)
    assert np.max(np.abs(gq)) < 1e-12 and np.max(np.abs(gk)) < 1e-12
    assert _rel_err(gv.sum(1), dout.sum(1)) < 1e-12


def pin_backward_linear_in_dout(orc):
    q, k, v = _rand(3040, 2, 15, 4, 3)
    d1, d2 = _rand(3041, 2, 15, 4, 3)[2], _rand(3042, 2, 15, 4, 3)[2]
    a = orc.causal_backward(q, k, v, 2.0 * d1 - 3.0 * d2)
    b1, b2 = orc.causal_backward(q, k, v, d1), orc.causal_backward(q, k, v, d2)
    for x, y1, y2 in zip(a, b1, b2):
        assert _rel_err(x, 2.0 * y1 - 3.0 * y2) < 1e-12


# ----------------------------------------------------------------------------
# Performer FAVOR+ features ("Linear Attention -- Math + Variants", Performer):
# phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m), E[phi(q) . phi(k)] = exp(q . k)
# ----------------------------------------------------------------------------
def pin_favor_unbiased_estimate(orc):
    """With m = 40000 Gaussian w_r the estimate phi(q) . phi(k) is within 5 standard
    errors of exp(q . k) (the standard error estimated from the same samples)."""
    rng = np.random.default_rng(4000)
    d, m = 8, 40000
    W = rng.standard_normal((m, d))
    for _ in range(3):
        q, k = rng.standard_normal(d) * 0.4, rng.standard_normal(d) * 0.4
        fq, fk = orc.favor_features(q[None], W)[0], orc.favor_features(k[None], W)[0]
        terms = fq * fk * m  # each term's mean is exp(q . k)
        est, se = terms.mean(), terms.std() / np.sqrt(m)
        assert abs(est - math.exp(float(q @ k))) < 5 * se, (est, math.exp(float(q @ k)), se)


def pin_favor_zero_projection(orc):
    """W = 0: every feature is exp(-|x|^2 / 2) / sqrt(m)."""
    x = np.array([[0.5, -1.0, 2.0], [0.0, 0.0, 0.0]])
    out = orc.favor_features(x, np.zeros((4, 3)))
    ref = np.exp(-0.5 * (x ** 2).sum(-1))[:, None] / 2.0 * np.ones((1, 4))
    assert _rel_err(out, ref) < 1e-15


def pin_favor_unit_projection(orc):
    """m = 1, w = e_1: phi(x) = exp(x_1 - |x|^2 / 2), with the library's exp."""
    x = np.array([[0.3, -0.2, 0.7, 1.1]])
    got = orc.favor_features(x, np.array([[1.0, 0.0, 0.0, 0.0]]))[0, 0]
    assert abs(got - math.exp(0.3 - 0.5 * (0.09 + 0.04 + 0.49 + 1.21))) < 1e-15


def pin_favor_coordinate_projections(orc):
    """Rows of W that pick single coordinates, in a non-square order (m = 2, d = 3):
    phi(x)_0 = exp(x_2 - |x|^2 / 2) / sqrt(2), phi(x)_1 = exp(-x_0 - |x|^2 / 2) / sqrt(2)."""
    x = np.array([[0.4, -0.3, 1.2], [-0.8, 0.5, 0.1]])
    W = np.array([[0.0, 0.0, 1.0], [-1.0, 0.0, 0.0]])
    got = orc.favor_features(x, W)
    for i in range(2):
        h = 0.5 * float(x[i] @ x[i])
        assert abs(got[i, 0] - math.exp(x[i, 2] - h) / math.sqrt(2.0)) < 1e-15
        assert abs(got[i, 1] - math.exp(-x[i, 0] - h) / math.sqrt(2.0)) < 1e-15


def pin_favor_positive_and_scale(orc):
    """Features are positive, and scaling m by 4 with repeated rows divides each by 2."""
    rng = np.random.default_rng(4010)
    x = rng.standard_normal((5, 6))
    W = rng.standard_normal((3, 6))
    a = orc.favor_features(x, W)
    b = orc.favor_features(x, np.tile(W, (4, 1)))
    assert np.all(a > 0) and _rel_err(b[:, :3], a / 2.0) < 1e-15


def pin_favor_attention_zero_projection(orc):
    """W = 0: phi(q) . phi(k) = exp(-|q|^2 / 2) exp(-|k|^2 / 2), so the query factor cancels
    and the FAVOR+ forms are the key-weighted averages o_i = sum_j a_j v_j / sum_j a_j with
    a_j = exp(-|k_j|^2 / 2), over j <= i (causal) or all j (non-causal)."""
    rng = np.random.default_rng(4020)
    N, d, dv, m = 9, 3, 2, 4
    q, k, v = rng.standard_normal((N, d)) * 0.5, rng.standard_normal((N, d)) * 0.5, rng.standard_normal((N, dv))
    W = np.zeros((m, d))
    a = np.exp(-0.5 * (k ** 2).sum(-1))
    causal = np.cumsum(a[:, None] * v, 0) / np.cumsum(a)[:, None]
    full = np.broadcast_to((a[:, None] * v).sum(0) / a.sum(), (N, dv))
    assert _rel_err(orc.causal_favor(q, k, v, W), causal) < 1e-14
    assert _rel_err(orc.noncausal_favor(q, k, v, W), full) < 1e-14


# ----------------------------------------------------------------------------
# Identities and special cases that reach the decode, prefix-state and backward
# forms from a second direction
# ----------------------------------------------------------------------------
def _phi_elu1(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def pin_backward_homogeneity(orc):
    """Where the clamp does not bind, o_i does not change when phi(q_i) is scaled, nor when
    every phi(k_j) is scaled by one factor, and o is linear in V.  By Euler's theorem on
    homogeneous functions: sum_r dphi(q_i)_r phi(q_i)_r = 0 for each i,
    sum_{j,r} dphi(k_j)_r phi(k_j)_r = 0, and sum_j v_j . dv_j = sum_i dO_i . o_i.  With
    dq = dphi(q) phi'(q), phi / phi' is x + 1 for x > 0 and 1 for x <= 0."""
    rng = np.random.default_rng(4030)
    N, dk, dv = 40, 5, 3
    q, k = rng.standard_normal((N, dk)), rng.standard_normal((N, dk))
    v, dout = rng.standard_normal((N, dv)), rng.standard_normal((N, dv))
    gq, gk, gv = orc.causal_backward(q, k, v, dout)

    def ratio(x):
        return np.where(x > 0, x + 1.0, 1.0)

    tq, tk = gq * ratio(q), gk * ratio(k)
    assert np.max(np.abs(tq.sum(-1))) <= 1e-12 * np.max(np.abs(tq).sum(-1))
    assert abs(tk.sum()) <= 1e-12 * np.abs(tk).sum()
    lhs, rhs = float((v * gv).sum()), float((dout * orc.causal_recurrent(q, k, v)).sum())
    assert abs(lhs - rhs) <= 1e-12 * max(abs(rhs), 1.0)


def pin_decode_from_zero_state_returns_v(orc):
    """From a zero state a step sees its own key only, so o = v for any q (the first-row case
    o_0 = v_0): the plain step, the decayed step for any gamma, and the general step."""
    rng = np.random.default_rng(4040)
    H, dk, dv = 3, 4, 2
    q, k, v = rng.standard_normal((H, dk)) * 0.5, rng.standard_normal((H, dk)) * 0.5, rng.standard_normal((H, dv))
    steps = [lambda S, z: orc.decode_step(S, z, q, k, v),
             lambda S, z: orc.decode_step_decay(S, z, q, k, v, np.array([0.0, 0.5, 1.0])),
             lambda S, z: orc.decode_step_general(S, z, q, k, v, fmap="relu", shift=0.5),
             lambda S, z: orc.decode_step_general(S, z, q, k, v, gamma=np.array([0.9, 0.5, 0.1]))]
    for step in steps:
        S, z = np.zeros((H, dk, dv)), np.zeros((H, dk))
        assert _rel_err(step(S, z), v) < 1e-14


def pin_decode_decay_zero_wipes_state(orc):
    """gamma = 0 forgets the state before the token: o = v from any state, decayed and general."""
    rng = np.random.default_rng(4050)
    H, dk, dv = 2, 3, 4
    q, k, v = rng.standard_normal((H, dk)) * 0.5, rng.standard_normal((H, dk)) * 0.5, rng.standard_normal((H, dv))
    for general in (False, True):
        S = np.ascontiguousarray(rng.standard_normal((H, dk, dv)))
        z = np.ascontiguousarray(np.abs(rng.standard_normal((H, dk))) + 1.0)
        o = (orc.decode_step_general(S, z, q, k, v, gamma=np.zeros(H)) if general
             else orc.decode_step_decay(S, z, q, k, v, np.zeros(H)))
        assert _rel_err(o, v) < 1e-14


def pin_decode_two_tokens_bruteforce(orc):
    """Two steps from a zero state against the two weights written out:
    o_1 = (g a_0 v_0 + a_1 v_1) / (g a_0 + a_1), a_j = phi(q_1) . phi(k_j), for elu + 1 (g = 1),
    ReLU + 1/4 and a decay g = 0.6."""
    rng = np.random.default_rng(4060)
    dk, dv = 3, 2
    q, k, v = rng.standard_normal((2, dk)), rng.standard_normal((2, dk)), rng.standard_normal((2, dv))
    cases = [("elu1", 0.0, None), ("relu", 0.25, None), ("elu1", 0.0, 0.6)]
    for fmap, shift, g in cases:
        phi = _phi_elu1 if fmap == "elu1" else (lambda x: np.maximum(x, 0.0) + shift)
        a = [float(phi(q[1]) @ phi(k[j])) for j in range(2)]
        w0 = a[0] * (1.0 if g is None else g)
        ref = (w0 * v[0] + a[1] * v[1]) / (w0 + a[1])
        S, z = np.zeros((1, dk, dv)), np.zeros((1, dk))
        gam = None if g is None else np.array([g])
        for t in range(2):
            o = orc.decode_step_general(S, z, q[t][None], k[t][None], v[t][None], gamma=gam, fmap=fmap,
                                        shift=shift)
        assert _rel_err(o[0], ref) < 1e-13, (fmap, g)


def pin_prefill_decay_zero_keeps_last_token(orc):
    """gamma = 0: after N tokens the state holds the last token only, S = phi(k)v^T, z = phi(k)."""
    rng = np.random.default_rng(4070)
    H, N, dk, dv = 2, 5, 3, 4
    k, v = rng.standard_normal((H, N, dk)), rng.standard_normal((H, N, dv))
    S, z = orc.prefill_state_general(k, v, gamma=np.zeros(H))
    fk = _phi_elu1(k[:, -1])
    assert _rel_err(S, fk[:, :, None] * v[:, -1][:, None, :]) < 1e-15
    assert _rel_err(z, fk) < 1e-15


def pin_bf16_known_values_first_row(orc):
    """bf16 bit patterns of known values reach the output unchanged through o_0 = v_0:
    0x3FC0 = 1.5, 0xC000 = -2.0, 0x3E20 = 0.15625, 0xBF80 = -1.0."""
    v = np.array([[[0x3FC0, 0xC000], [0x3E20, 0xBF80]]], dtype=np.uint16)  # [1, N=2, dv=2]
    qk = np.array([[[0x3F80], [0x3F00]]], dtype=np.uint16)                 # 1.0 and 0.5, dk = 1
    o = orc.causal_recurrent(qk, qk, v, EPS)
    assert o[0, 0, 0] == 1.5 and o[0, 0, 1] == -2.0


def pin_decay_quadratic_forms(orc):
    """The decayed quadratic companion form: gamma = 0 keeps only the current token
    (o = v), and for gamma in (0, 1) it agrees with the decayed recurrence."""
    q, k, v = _rand(1080, 2, 25, 3, 2)
    assert _rel_err(orc.causal_decay_quadratic(q, k, v, np.zeros(2), EPS), v) < 1e-14
    g = np.array([0.7, 0.95])
    assert _rel_err(orc.causal_decay_quadratic(q, k, v, g, EPS), orc.causal_decay_recurrent(q, k, v, g, EPS)) < 1e-12


# ----------------------------------------------------------------------------
# gated state, one gate per key feature ("Linear Attention", What is actually lost:
# S_t = G_t (.) S_{t-1} + phi(k_t) v_t^T; "Linear Attention -- Math + Variants",
# RetNet and gated linear attention: S_i = Diag(alpha_i) S_{i-1} + k_i v_i^T)
# ----------------------------------------------------------------------------
def gated_pairwise_np(q, k, v, alpha, eps=EPS):
    """w_ij = sum_r phi(q_i)[r] phi(k_j)[r] prod_{s=j+1..i} alpha_s[r] for j <= i, by
    cumulative sums of log(alpha) in numpy (a gate of 0 handled by counting zeros),
    o_i = sum_j w_ij v_j / max(sum_j w_ij, eps).  Dense, float64."""
    fq, fk = phi_np(q), phi_np(k)
    a = np.asarray(alpha, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    zero = (a == 0.0)
    la = np.log(np.where(zero, 1.0, a))
    L = np.cumsum(la, axis=-2)                      # L_i = sum_{s<=i} log alpha_s
    Z = np.cumsum(zero, axis=-2)                    # zeros among alpha_0..alpha_i
    N = q.shape[-2]
    out = np.empty(q.shape[:-1] + (v.shape[-1],))
    for i in range(N):
        # prod_{s=j+1..i} alpha_s = exp(L_i - L_j), zero if a gate in (j, i] is zero
        dec = np.exp(L[..., i:i + 1, :] - L[..., :i + 1, :])
        dec = np.where((Z[..., i:i + 1, :] - Z[..., :i + 1, :]) > 0, 0.0, dec)
        w = np.einsum("...r,...jr->...j", fq[..., i, :], fk[..., :i + 1, :] * dec)
        den = np.maximum(w.sum(-1, keepdims=True), eps)
        out[..., i, :] = np.einsum("...j,...jc->...c", w, v[..., :i + 1, :]) / den
    return out


def _gate(seed, shape, lo=0.3):
    return np.random.default_rng(seed).uniform(lo, 1.0, size=shape)


def pin_gated_equals_numpy_pairwise(orc):
    """The gated recurrence and the oracle's own pairwise form equal the numpy form
    above (dk != dv; gates in [0.3, 1), a few exactly 0 and 1)."""
    q, k, v = _rand(1100, 3, 40, 5, 3)
    a = _gate(1101, k.shape)
    a[0, 7, :] = 0.0
    a[1, 3, 2] = 0.0
    a[2, :, 4] = 1.0
    ref = gated_pairwise_np(q, k, v, a)
    assert _rel_err(orc.causal_gated_recurrent(q, k, v, a, EPS), ref) < 1e-12
    assert _rel_err(orc.causal_gated_quadratic(q, k, v, a, EPS), ref) < 1e-12


def pin_gated_constant_gate_is_scalar_decay(orc):
    """alpha_t[r] = gamma for every token and feature reduces to the (pinned) scalar
    decay of each head."""
    q, k, v = _rand(1110, 4, 30, 4, 6)
    g = np.array([1.0, 0.9, 0.5, 0.0])
    a = np.broadcast_to(g[:, None, None], k.shape)
    assert _rel_err(orc.causal_gated_recurrent(q, k, v, a, EPS), orc.causal_decay_recurrent(q, k, v, g, EPS)) < 1e-13


def pin_gated_one_is_undecayed_and_zero_returns_v(orc):
    q, k, v = _rand(1120, 2, 25, 5, 4)
    assert _rel_err(orc.causal_gated_recurrent(q, k, v, np.ones(k.shape), EPS),
                    pairwise_bruteforce(q, k, v, causal=True)) < 1e-12
    assert _rel_err(orc.causal_gated_recurrent(q, k, v, np.zeros(k.shape), EPS), v) < 1e-14


def pin_gated_exact_rational(orc):
    """Tiny inputs with q, k > 0 (phi = x + 1 exact) and gates in {1/4, 1/2, 3/4, 1},
    one per (token, feature), against exact rational arithmetic of the unrolled form."""
    rng = np.random.default_rng(1130)
    N, dk, dv = 6, 3, 2
    qv = rng.integers(1, 8, size=(N, dk)) / 8.0
    kv = rng.integers(1, 8, size=(N, dk)) / 8.0
    vv = rng.integers(-8, 9, size=(N, dv)) / 4.0
    av = rng.integers(1, 5, size=(N, dk)) / 4.0
    got = orc.causal_gated_recurrent(qv[None], kv[None], vv[None], av[None], 0.0)[0]
    fr = lambda x: Fraction(x).limit_denominator(64)
    fq = [[fr(x) + 1 for x in row] for row in qv]
    fk = [[fr(x) + 1 for x in row] for row in kv]
    vf = [[fr(x) for x in row] for row in vv]
    af = [[fr(x) for x in row] for row in av]
    for i in range(N):
        num = [Fraction(0)] * dv
        den = Fraction(0)
        for j in range(i + 1):
            w = Fraction(0)
            for r in range(dk):
                p = Fraction(1)
                for s_ in range(j + 1, i + 1):
                    p *= af[s_][r]
                w += fq[i][r] * fk[j][r] * p
            den += w
            for c in range(dv):
                num[c] += w * vf[j][c]
        for c in range(dv):
            assert abs(got[i, c] - float(num[c] / den)) <= 1e-14 * max(1.0, abs(float(num[c] / den)))


def pin_gated_gate_acts_per_key_feature(orc):
    """A gate that closes feature 0 only (alpha[:, 0] = 0, the rest 1) leaves the
    other features' history untouched: the output equals the ungated form computed
    with feature 0 of every earlier key removed from the weights."""
    q, k, v = _rand(1140, 2, 20, 4, 3)
    a = np.ones(k.shape)
    a[..., 0] = 0.0
    fq, fk = phi_np(q), phi_np(k)
    N = q.shape[-2]
    ref = np.empty(v.shape)
    for i in range(N):
        w = np.einsum("br,bjr->bj", fq[:, i, 1:], fk[:, :i + 1, 1:])
        w[:, i] += fq[:, i, 0] * fk[:, i, 0]           # feature 0 of the current key only
        ref[:, i] = np.einsum("bj,bjc->bc", w, v[:, :i + 1]) / np.maximum(w.sum(-1), EPS)[:, None]
    assert _rel_err(orc.causal_gated_recurrent(q, k, v, a, EPS), ref) < 1e-12


def pin_gated_decode_and_prefill_continue_causal(orc):
    """Gated decode steps from a zero state reproduce the gated causal forward at
    every position; the gated prefill state over a prefix, continued by decode
    steps, does too; and the prefill state equals the numpy sum of its terms."""
    BH, N, P, dk, dv = 3, 18, 7, 5, 4
    q, k, v = _rand(1150, BH, N, dk, dv)
    a = _gate(1151, k.shape)
    full = gated_pairwise_np(q, k, v, a)
    S = np.zeros((BH, dk, dv))
    z = np.zeros((BH, dk))
    for t in range(N):
        o = orc.decode_step_gated(S, z, q[:, t], k[:, t], v[:, t], a[:, t], EPS)
        assert _rel_err(o, full[:, t]) < 1e-12, t
    S, z = orc.prefill_state_gated(k[:, :P], v[:, :P], a[:, :P])
    fk = phi_np(k[:, :P])
    dec = np.ones((BH, P, dk))
    for t in range(P):
        dec[:, t] = np.prod(a[:, t + 1:P], axis=1)
    assert _rel_err(S, np.einsum("btr,btc->brc", fk * dec, v[:, :P])) < 1e-12
    assert _rel_err(z, (fk * dec).sum(1)) < 1e-12
    for t in range(P, N):
        o = orc.decode_step_gated(S, z, q[:, t], k[:, t], v[:, t], a[:, t], EPS)
        assert _rel_err(o, full[:, t]) < 1e-12, t


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
