/*
 * Float64 CPU oracle for causal kernelized (linear) attention, phi(x)=elu(x)+1.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline / reference arm may load or run this library.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * Plain loops in double precision, one (batch, head) sequence at a time; the
 * only parallelism is OpenMP across independent (b,h) sequences, which does not
 * change any result.  Every form below follows one passage of the pages:
 *
 *   [wiki]     "Linear Attention", aiwiki.thehackersbrain.dev
 *   [learn]    "Linear attention", learn.pranaymahendrakar.com
 *   [problems] "26. Linear (Kernelized) Attention: A Softmax-Free Alternative"
 *   [mlblogg]  "Linear attention: change the order.", mlblogg.com
 *   [math]     "Linear Attention -- Math + Variants", aicassindra.com
 *
 * Readings taken where the pages differ or are silent:
 *   - normaliser: o = num / max(den, eps) (the clamp of the [wiki] chunked
 *     listing); the "+1e-6" of [learn]/[problems] and "clip(1e-8)" of [mlblogg]
 *     agree with it to < 1e-7 relative whenever den >> eps;
 *   - phi(x) = x + 1 for x > 0, exp(x) otherwise: elu with alpha = 1 plus one,
 *     written in the overflow-free way of the [mlblogg] implementation section;
 *   - causality is inclusive (token i sees keys j <= i): update, then read
 *     ([mlblogg] "The causal recurrence"; [learn] Developer listing);
 *   - no 1/sqrt(d) scaling of q or k (only softmax scales, [math]);
 *   - state and all arithmetic in double; inputs are given as float64,
 *     float32 or bf16 bit patterns and widened exactly;
 *   - variants (the *_general forms): the decay, the ReLU and identity-plus-
 *     shift feature maps and the normaliser-free output compose freely; the
 *     decayed normaliser z decays with the same gamma as S.
 *
 * Tensor layouts (row-major, contiguous):
 *   q, k [BH, N, dk];  v, o [BH, N, dv];  S [BH, dk, dv];  z [BH, dk].
 * Input element type code: 0 = float64, 1 = float32, 2 = bf16 (uint16 bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F64 0
#define ORACLE_F32 1
#define ORACLE_BF16 2

/* Read element i of an input array of the given type as a double. */
static double load(const void *p, int type, int64_t i)
{
    if (type == ORACLE_F64)
        return ((const double *)p)[i];
    if (type == ORACLE_F32)
        return (double)((const float *)p)[i];
    /* bf16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* phi(x) = elu(x) + 1 with alpha = 1 ([math] "Linear Transformer: elu+1";
 * [wiki] listing applies F.elu then adds one; [mlblogg] writes the same map as
 * where(x >= 0, x + 1, exp(min(x, 0)))).  Both branches give 1 at x = 0. */
double la_oracle_phi(double x)
{
    return x > 0.0 ? x + 1.0 : exp(x);
}

static double clamp_den(double den, double eps)
{
    return den > eps ? den : eps;
}

/* phi of row t of a [N, d] slice starting at element `base`. */
static void phi_row(const void *x, int type, int64_t base, int t, int d, double *out)
{
    for (int c = 0; c < d; ++c)
        out[c] = la_oracle_phi(load(x, type, base + (int64_t)t * d + c));
}

/* ---------------------------------------------------------------------------
 * Causal recurrence, token by token: the defining form.
 * [learn] Researcher "Derivation": S_i = S_{i-1} + phi(k_i) v_i^T,
 * z_i = z_{i-1} + phi(k_i), o_i = S_i^T phi(q_i) / z_i^T phi(q_i);
 * [problems] Step-by-Step steps 2-5 (state update before the read).
 * ------------------------------------------------------------------------- */
void la_oracle_causal_recurrent(const void *q, const void *k, const void *v, int type,
                                double *o, int BH, int N, int dk, int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        double *S = calloc((size_t)dk * dv, sizeof(double));
        double *z = calloc((size_t)dk, sizeof(double));
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        double *vt = malloc(sizeof(double) * dv);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int t = 0; t < N; ++t) {
            phi_row(q, type, qb, t, dk, fq);
            phi_row(k, type, qb, t, dk, fk);
            for (int c = 0; c < dv; ++c)
                vt[c] = load(v, type, vb + (int64_t)t * dv + c);
            /* S += phi(k_t) v_t^T ; z += phi(k_t) */
            for (int r = 0; r < dk; ++r) {
                double *Sr = S + (size_t)r * dv;
                for (int c = 0; c < dv; ++c)
                    Sr[c] += fk[r] * vt[c];
                z[r] += fk[r];
            }
            /* o_t = phi(q_t)^T S / max(phi(q_t)^T z, eps) */
            double den = 0.0;
            for (int r = 0; r < dk; ++r)
                den += fq[r] * z[r];
            double *ot = o + vb + (int64_t)t * dv;
            for (int c = 0; c < dv; ++c)
                ot[c] = 0.0;
            for (int r = 0; r < dk; ++r) {
                const double *Sr = S + (size_t)r * dv;
                for (int c = 0; c < dv; ++c)
                    ot[c] += fq[r] * Sr[c];
            }
            den = clamp_den(den, eps);
            for (int c = 0; c < dv; ++c)
                ot[c] /= den;
        }
        free(S); free(z); free(fq); free(fk); free(vt);
    }
}

/* ---------------------------------------------------------------------------
 * Chunked parallel form ([wiki] listing "linear_attention_chunked"): for each
 * chunk, inter = phi(Q_c) state_before, intra = tril(phi(Q_c) phi(K_c)^T) V_c,
 * denominator = phi(Q_c) z_before + row sums of the masked scores, then the
 * state and z absorb the chunk.  The last chunk may be shorter than `chunk`.
 * ------------------------------------------------------------------------- */
void la_oracle_causal_chunked(const void *q, const void *k, const void *v, int type,
                              double *o, int BH, int N, int dk, int dv, int chunk,
                              double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        double *state = calloc((size_t)dk * dv, sizeof(double));
        double *z = calloc((size_t)dk, sizeof(double));
        double *fq = malloc(sizeof(double) * dk);
        double *fkj = malloc(sizeof(double) * dk);
        double *num = malloc(sizeof(double) * dv);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int i0 = 0; i0 < N; i0 += chunk) {
            int len = N - i0 < chunk ? N - i0 : chunk;
            for (int a = 0; a < len; ++a) {
                phi_row(q, type, qb, i0 + a, dk, fq);
                /* inter: phi(q) @ state (state holds earlier chunks only) */
                for (int c = 0; c < dv; ++c) {
                    double s = 0.0;
                    for (int r = 0; r < dk; ++r)
                        s += fq[r] * state[(size_t)r * dv + c];
                    num[c] = s;
                }
                double den = 0.0;
                for (int r = 0; r < dk; ++r)
                    den += fq[r] * z[r];
                /* intra: masked scores, keys b <= a of this chunk */
                for (int b = 0; b <= a; ++b) {
                    phi_row(k, type, qb, i0 + b, dk, fkj);
                    double s = 0.0;
                    for (int r = 0; r < dk; ++r)
                        s += fq[r] * fkj[r];
                    for (int c = 0; c < dv; ++c)
                        num[c] += s * load(v, type, vb + (int64_t)(i0 + b) * dv + c);
                    den += s;
                }
                den = clamp_den(den, eps);
                for (int c = 0; c < dv; ++c)
                    o[vb + (int64_t)(i0 + a) * dv + c] = num[c] / den;
            }
            /* state += phi(K_c)^T V_c ; z += column sums of phi(K_c) */
            for (int b = 0; b < len; ++b) {
                phi_row(k, type, qb, i0 + b, dk, fkj);
                for (int r = 0; r < dk; ++r) {
                    for (int c = 0; c < dv; ++c)
                        state[(size_t)r * dv + c] +=
                            fkj[r] * load(v, type, vb + (int64_t)(i0 + b) * dv + c);
                    z[r] += fkj[r];
                }
            }
        }
        free(state); free(z); free(fq); free(fkj); free(num);
    }
}

/* ---------------------------------------------------------------------------
 * Masked quadratic form ([learn] Developer listing, part 3; [problems] Key
 * Functions, the directly-masked score matrix): scores = phi(Q) phi(K)^T kept
 * for j <= i, o = scores V / row sums.  O(N^2): cross-check only.
 * ------------------------------------------------------------------------- */
void la_oracle_causal_quadratic(const void *q, const void *k, const void *v, int type,
                                double *o, int BH, int N, int dk, int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int i = 0; i < N; ++i) {
            phi_row(q, type, qb, i, dk, fq);
            double *oi = o + vb + (int64_t)i * dv;
            for (int c = 0; c < dv; ++c)
                oi[c] = 0.0;
            double rowsum = 0.0;
            for (int j = 0; j <= i; ++j) {
                phi_row(k, type, qb, j, dk, fk);
                double s = 0.0;
                for (int r = 0; r < dk; ++r)
                    s += fq[r] * fk[r];
                rowsum += s;
                for (int c = 0; c < dv; ++c)
                    oi[c] += s * load(v, type, vb + (int64_t)j * dv + c);
            }
            rowsum = clamp_den(rowsum, eps);
            for (int c = 0; c < dv; ++c)
                oi[c] /= rowsum;
        }
        free(fq); free(fk);
    }
}

/* ---------------------------------------------------------------------------
 * Final state of a prefix: S = sum_t phi(k_t) v_t^T, z = sum_t phi(k_t) over
 * all N tokens ([math] "The quadratic wall": S and z; [problems] step 3).
 * ------------------------------------------------------------------------- */
void la_oracle_prefill_state(const void *k, const void *v, int type, double *S, double *z,
                             int BH, int N, int dk, int dv)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * dk * dv;
        double *zb = z + (size_t)bh * dk;
        double *fk = malloc(sizeof(double) * dk);
        const int64_t kb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (size_t e = 0; e < (size_t)dk * dv; ++e)
            Sb[e] = 0.0;
        for (int r = 0; r < dk; ++r)
            zb[r] = 0.0;
        for (int t = 0; t < N; ++t) {
            phi_row(k, type, kb, t, dk, fk);
            for (int r = 0; r < dk; ++r) {
                for (int c = 0; c < dv; ++c)
                    Sb[(size_t)r * dv + c] += fk[r] * load(v, type, vb + (int64_t)t * dv + c);
                zb[r] += fk[r];
            }
        }
        free(fk);
    }
}

/* ---------------------------------------------------------------------------
 * Non-causal associative form ([mlblogg] "An implementation you can check":
 * state = phi(K)^T V, normalizer = sum phi(K), o = phi(Q) state / phi(Q) normalizer;
 * [math] o_i = phi(q_i)^T S / phi(q_i)^T z with S, z summed over all j).
 * ------------------------------------------------------------------------- */
void la_oracle_noncausal(const void *q, const void *k, const void *v, int type,
                         double *o, int BH, int N, int dk, int dv, double eps)
{
    double *S = malloc(sizeof(double) * (size_t)BH * dk * dv);
    double *z = malloc(sizeof(double) * (size_t)BH * dk);
    la_oracle_prefill_state(k, v, type, S, z, BH, N, dk, dv);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        const double *Sb = S + (size_t)bh * dk * dv;
        const double *zb = z + (size_t)bh * dk;
        double *fq = malloc(sizeof(double) * dk);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int i = 0; i < N; ++i) {
            phi_row(q, type, qb, i, dk, fq);
            double den = 0.0;
            for (int r = 0; r < dk; ++r)
                den += fq[r] * zb[r];
            den = clamp_den(den, eps);
            double *oi = o + vb + (int64_t)i * dv;
            for (int c = 0; c < dv; ++c) {
                double s = 0.0;
                for (int r = 0; r < dk; ++r)
                    s += fq[r] * Sb[(size_t)r * dv + c];
                oi[c] = s / den;
            }
        }
        free(fq);
    }
    free(S); free(z);
}

/* ---------------------------------------------------------------------------
 * Brute-force pairwise non-causal form ([mlblogg] check: pairwise =
 * phi(q) phi(k)^T, reference = pairwise v / row sums).  O(N^2): cross-check.
 * ------------------------------------------------------------------------- */
void la_oracle_noncausal_pairwise(const void *q, const void *k, const void *v, int type,
                                  double *o, int BH, int N, int dk, int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int i = 0; i < N; ++i) {
            phi_row(q, type, qb, i, dk, fq);
            double *oi = o + vb + (int64_t)i * dv;
            for (int c = 0; c < dv; ++c)
                oi[c] = 0.0;
            double rowsum = 0.0;
            for (int j = 0; j < N; ++j) {
                phi_row(k, type, qb, j, dk, fk);
                double s = 0.0;
                for (int r = 0; r < dk; ++r)
                    s += fq[r] * fk[r];
                rowsum += s;
                for (int c = 0; c < dv; ++c)
                    oi[c] += s * load(v, type, vb + (int64_t)j * dv + c);
            }
            rowsum = clamp_den(rowsum, eps);
            for (int c = 0; c < dv; ++c)
                oi[c] /= rowsum;
        }
        free(fq); free(fk);
    }
}

/* ---------------------------------------------------------------------------
 * One recurrent decode step for BH independent heads, state in place
 * ([wiki] "It is a linear RNN": O(d^2) per token; [learn] Developer listing,
 * part 2, loop body; [problems] steps 3-4).  q, k [BH, dk], v [BH, dv],
 * S [BH, dk, dv] and z [BH, dk] double, o [BH, dv] double.
 * ------------------------------------------------------------------------- */
void la_oracle_decode_step(double *S, double *z, const void *q, const void *k,
                           const void *v, int type, double *o, int BH, int dk, int dv,
                           double eps)
{
#pragma omp parallel for schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * dk * dv;
        double *zb = z + (size_t)bh * dk;
        double *ob = o + (size_t)bh * dv;
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        for (int r = 0; r < dk; ++r) {
            fq[r] = la_oracle_phi(load(q, type, (int64_t)bh * dk + r));
            fk[r] = la_oracle_phi(load(k, type, (int64_t)bh * dk + r));
        }
        for (int r = 0; r < dk; ++r) {
            for (int c = 0; c < dv; ++c)
                Sb[(size_t)r * dv + c] += fk[r] * load(v, type, (int64_t)bh * dv + c);
            zb[r] += fk[r];
        }
        double den = 0.0;
        for (int r = 0; r < dk; ++r)
            den += fq[r] * zb[r];
        den = clamp_den(den, eps);
        for (int c = 0; c < dv; ++c) {
            double s = 0.0;
            for (int r = 0; r < dk; ++r)
                s += fq[r] * Sb[(size_t)r * dv + c];
            ob[c] = s / den;
        }
        free(fq); free(fk);
    }
}

/* ---------------------------------------------------------------------------
 * Decayed state (scalar decay per sequence).  [math] "RetNet and gated linear
 * attention: decay in the state": S_i = gamma S_{i-1} + k_i v_i^T with a fixed
 * per-head gamma; [wiki] "What is actually lost": S_t = G_t (.) S_{t-1} +
 * phi(k_t) v_t^T; [learn] "Try it yourself": S = 0.9 * S + outer(k_t, v_t).
 * Reading: phi as above, and the normaliser z decays with the same gamma, so
 * gamma = 1 is the undecayed form above:
 *   S_t = g S_{t-1} + phi(k_t) v_t^T,  z_t = g z_{t-1} + phi(k_t),
 *   o_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps).
 * gamma: one value per (b,h) sequence, [BH] double.
 * ------------------------------------------------------------------------- */
void la_oracle_causal_decay_recurrent(const void *q, const void *k, const void *v, int type,
                                      const double *gamma, double *o, int BH, int N, int dk,
                                      int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        const double g = gamma[bh];
        double *S = calloc((size_t)dk * dv, sizeof(double));
        double *z = calloc((size_t)dk, sizeof(double));
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        double *vt = malloc(sizeof(double) * dv);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int t = 0; t < N; ++t) {
            phi_row(q, type, qb, t, dk, fq);
            phi_row(k, type, qb, t, dk, fk);
            for (int c = 0; c < dv; ++c)
                vt[c] = load(v, type, vb + (int64_t)t * dv + c);
            /* S = g S + phi(k_t) v_t^T ; z = g z + phi(k_t) */
            for (int r = 0; r < dk; ++r) {
                double *Sr = S + (size_t)r * dv;
                for (int c = 0; c < dv; ++c)
                    Sr[c] = g * Sr[c] + fk[r] * vt[c];
                z[r] = g * z[r] + fk[r];
            }
            double den = 0.0;
            for (int r = 0; r < dk; ++r)
                den += fq[r] * z[r];
            double *ot = o + vb + (int64_t)t * dv;
            for (int c = 0; c < dv; ++c)
                ot[c] = 0.0;
            for (int r = 0; r < dk; ++r) {
                const double *Sr = S + (size_t)r * dv;
                for (int c = 0; c < dv; ++c)
                    ot[c] += fq[r] * Sr[c];
            }
            den = clamp_den(den, eps);
            for (int c = 0; c < dv; ++c)
                ot[c] /= den;
        }
        free(S); free(z); free(fq); free(fk); free(vt);
    }
}

/* The weighted quadratic form the decayed recurrence equals ([learn] "Try it
 * yourself": the weighted quadratic form it does match): scores
 * g^(i-j) phi(q_i).phi(k_j) kept for j <= i, o = scores V / row sums.  O(N^2):
 * cross-check only.  0^0 = 1 (the token itself). */
void la_oracle_causal_decay_quadratic(const void *q, const void *k, const void *v, int type,
                                      const double *gamma, double *o, int BH, int N, int dk,
                                      int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        const double g = gamma[bh];
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int i = 0; i < N; ++i) {
            phi_row(q, type, qb, i, dk, fq);
            double *oi = o + vb + (int64_t)i * dv;
            for (int c = 0; c < dv; ++c)
                oi[c] = 0.0;
            double rowsum = 0.0;
            for (int j = 0; j <= i; ++j) {
                phi_row(k, type, qb, j, dk, fk);
                double s = 0.0;
                for (int r = 0; r < dk; ++r)
                    s += fq[r] * fk[r];
                s *= (i == j) ? 1.0 : pow(g, (double)(i - j));
                rowsum += s;
                for (int c = 0; c < dv; ++c)
                    oi[c] += s * load(v, type, vb + (int64_t)j * dv + c);
            }
            rowsum = clamp_den(rowsum, eps);
            for (int c = 0; c < dv; ++c)
                oi[c] /= rowsum;
        }
        free(fq); free(fk);
    }
}

/* One decayed decode step, state in place: S = g S + phi(k) v^T, z = g z +
 * phi(k), then o = phi(q)^T S / max(phi(q)^T z, eps).  gamma [BH]. */
void la_oracle_decode_step_decay(double *S, double *z, const void *q, const void *k,
                                 const void *v, int type, const double *gamma, double *o, int BH,
                                 int dk, int dv, double eps)
{
#pragma omp parallel for schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        const double g = gamma[bh];
        double *Sb = S + (size_t)bh * dk * dv;
        double *zb = z + (size_t)bh * dk;
        double *ob = o + (size_t)bh * dv;
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        for (int r = 0; r < dk; ++r) {
            fq[r] = la_oracle_phi(load(q, type, (int64_t)bh * dk + r));
            fk[r] = la_oracle_phi(load(k, type, (int64_t)bh * dk + r));
        }
        for (int r = 0; r < dk; ++r) {
            for (int c = 0; c < dv; ++c)
                Sb[(size_t)r * dv + c] = g * Sb[(size_t)r * dv + c] + fk[r] * load(v, type, (int64_t)bh * dv + c);
            zb[r] = g * zb[r] + fk[r];
        }
        double den = 0.0;
        for (int r = 0; r < dk; ++r)
            den += fq[r] * zb[r];
        den = clamp_den(den, eps);
        for (int c = 0; c < dv; ++c) {
            double s = 0.0;
            for (int r = 0; r < dk; ++r)
                s += fq[r] * Sb[(size_t)r * dv + c];
            ob[c] = s / den;
        }
        free(fq); free(fk);
    }
}

/* ---------------------------------------------------------------------------
 * Variants of the feature map and of the normaliser, for every form above.
 *
 * Feature maps ([learn] "What the pieces are for": ReLU among the other
 * choices; [math] "Feature-map families": ReLU and identity-plus-shift;
 * [problems] "Key Functions & Tricks": relu(x) + eps):
 *   map 0: elu(x) + 1 (the default; the shift is ignored),
 *   map 1: max(x, 0) + c,
 *   map 2: x + c.
 * Normaliser ([math] "Implementation reality": most variants drop phi(q)^T z
 * and normalise the output with a layer after attention): normalize = 1 gives
 * o = phi(q)^T S / max(phi(q)^T z, eps); normalize = 0 gives o = phi(q)^T S.
 * gamma: NULL for no decay, else [BH] (the decayed state above).
 * ------------------------------------------------------------------------- */
static double phi_map(double x, int map, double c)
{
    if (map == 1)
        return (x > 0.0 ? x : 0.0) + c;
    if (map == 2)
        return x + c;
    return la_oracle_phi(x);
}

static void phi_row_map(const void *x, int type, int64_t base, int t, int d, int map, double c, double *out)
{
    for (int i = 0; i < d; ++i)
        out[i] = phi_map(load(x, type, base + (int64_t)t * d + i), map, c);
}

/* The recurrence with a feature map, an optional decay and an optional normaliser. */
void la_oracle_causal_general(const void *q, const void *k, const void *v, int type,
                              const double *gamma, int map, double shift, int normalize,
                              double *o, int BH, int N, int dk, int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        const double g = gamma ? gamma[bh] : 1.0;
        double *S = calloc((size_t)dk * dv, sizeof(double));
        double *z = calloc((size_t)dk, sizeof(double));
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        double *vt = malloc(sizeof(double) * dv);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int t = 0; t < N; ++t) {
            phi_row_map(q, type, qb, t, dk, map, shift, fq);
            phi_row_map(k, type, qb, t, dk, map, shift, fk);
            for (int c = 0; c < dv; ++c)
                vt[c] = load(v, type, vb + (int64_t)t * dv + c);
            for (int r = 0; r < dk; ++r) {
                double *Sr = S + (size_t)r * dv;
                for (int c = 0; c < dv; ++c)
                    Sr[c] = g * Sr[c] + fk[r] * vt[c];
                z[r] = g * z[r] + fk[r];
            }
            double *ot = o + vb + (int64_t)t * dv;
            for (int c = 0; c < dv; ++c)
                ot[c] = 0.0;
            for (int r = 0; r < dk; ++r) {
                const double *Sr = S + (size_t)r * dv;
                for (int c = 0; c < dv; ++c)
                    ot[c] += fq[r] * Sr[c];
            }
            if (normalize) {
                double den = 0.0;
                for (int r = 0; r < dk; ++r)
                    den += fq[r] * z[r];
                den = clamp_den(den, eps);
                for (int c = 0; c < dv; ++c)
                    ot[c] /= den;
            }
        }
        free(S); free(z); free(fq); free(fk); free(vt);
    }
}

/* The same function as masked (and weighted) scores: s_ij = g^(i-j)
 * phi(q_i).phi(k_j) for j <= i; o = s V, divided by the row sums when
 * normalize.  O(N^2): cross-check only. */
void la_oracle_causal_general_quadratic(const void *q, const void *k, const void *v, int type,
                                        const double *gamma, int map, double shift, int normalize,
                                        double *o, int BH, int N, int dk, int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        const double g = gamma ? gamma[bh] : 1.0;
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int i = 0; i < N; ++i) {
            phi_row_map(q, type, qb, i, dk, map, shift, fq);
            double *oi = o + vb + (int64_t)i * dv;
            for (int c = 0; c < dv; ++c)
                oi[c] = 0.0;
            double rowsum = 0.0;
            for (int j = 0; j <= i; ++j) {
                phi_row_map(k, type, qb, j, dk, map, shift, fk);
                double s = 0.0;
                for (int r = 0; r < dk; ++r)
                    s += fq[r] * fk[r];
                s *= (i == j) ? 1.0 : pow(g, (double)(i - j));
                rowsum += s;
                for (int c = 0; c < dv; ++c)
                    oi[c] += s * load(v, type, vb + (int64_t)j * dv + c);
            }
            if (normalize) {
                rowsum = clamp_den(rowsum, eps);
                for (int c = 0; c < dv; ++c)
                    oi[c] /= rowsum;
            }
        }
        free(fq); free(fk);
    }
}

/* Prefix state under a feature map and an optional decay: S = sum_t
 * g^(N-1-t) phi(k_t) v_t^T, z likewise (the recurrence from a zero state). */
void la_oracle_prefill_state_general(const void *k, const void *v, int type, const double *gamma,
                                     int map, double shift, double *S, double *z, int BH, int N,
                                     int dk, int dv)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        const double g = gamma ? gamma[bh] : 1.0;
        double *Sb = S + (size_t)bh * dk * dv;
        double *zb = z + (size_t)bh * dk;
        double *fk = malloc(sizeof(double) * dk);
        const int64_t kb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (size_t e = 0; e < (size_t)dk * dv; ++e)
            Sb[e] = 0.0;
        for (int r = 0; r < dk; ++r)
            zb[r] = 0.0;
        for (int t = 0; t < N; ++t) {
            phi_row_map(k, type, kb, t, dk, map, shift, fk);
            for (int r = 0; r < dk; ++r) {
                for (int c = 0; c < dv; ++c)
                    Sb[(size_t)r * dv + c] = g * Sb[(size_t)r * dv + c] +
                                             fk[r] * load(v, type, vb + (int64_t)t * dv + c);
                zb[r] = g * zb[r] + fk[r];
            }
        }
        free(fk);
    }
}

/* Non-causal form under a feature map, with or without the normaliser. */
void la_oracle_noncausal_general(const void *q, const void *k, const void *v, int type, int map,
                                 double shift, int normalize, double *o, int BH, int N, int dk,
                                 int dv, double eps)
{
    double *S = malloc(sizeof(double) * (size_t)BH * dk * dv);
    double *z = malloc(sizeof(double) * (size_t)BH * dk);
    la_oracle_prefill_state_general(k, v, type, NULL, map, shift, S, z, BH, N, dk, dv);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        const double *Sb = S + (size_t)bh * dk * dv;
        const double *zb = z + (size_t)bh * dk;
        double *fq = malloc(sizeof(double) * dk);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int i = 0; i < N; ++i) {
            phi_row_map(q, type, qb, i, dk, map, shift, fq);
            double den = 1.0;
            if (normalize) {
                den = 0.0;
                for (int r = 0; r < dk; ++r)
                    den += fq[r] * zb[r];
                den = clamp_den(den, eps);
            }
            double *oi = o + vb + (int64_t)i * dv;
            for (int c = 0; c < dv; ++c) {
                double s = 0.0;
                for (int r = 0; r < dk; ++r)
                    s += fq[r] * Sb[(size_t)r * dv + c];
                oi[c] = normalize ? s / den : s;
            }
        }
        free(fq);
    }
    free(S); free(z);
}

/* One decode step under a feature map, an optional decay and an optional
 * normaliser: S = g S + phi(k) v^T, z = g z + phi(k), then the read. */
void la_oracle_decode_step_general(double *S, double *z, const void *q, const void *k, const void *v,
                                   int type, const double *gamma, int map, double shift, int normalize,
                                   double *o, int BH, int dk, int dv, double eps)
{
#pragma omp parallel for schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        const double g = gamma ? gamma[bh] : 1.0;
        double *Sb = S + (size_t)bh * dk * dv;
        double *zb = z + (size_t)bh * dk;
        double *ob = o + (size_t)bh * dv;
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        for (int r = 0; r < dk; ++r) {
            fq[r] = phi_map(load(q, type, (int64_t)bh * dk + r), map, shift);
            fk[r] = phi_map(load(k, type, (int64_t)bh * dk + r), map, shift);
        }
        for (int r = 0; r < dk; ++r) {
            for (int c = 0; c < dv; ++c)
                Sb[(size_t)r * dv + c] = g * Sb[(size_t)r * dv + c] + fk[r] * load(v, type, (int64_t)bh * dv + c);
            zb[r] = g * zb[r] + fk[r];
        }
        double den = 1.0;
        if (normalize) {
            den = 0.0;
            for (int r = 0; r < dk; ++r)
                den += fq[r] * zb[r];
            den = clamp_den(den, eps);
        }
        for (int c = 0; c < dv; ++c) {
            double s = 0.0;
            for (int r = 0; r < dk; ++r)
                s += fq[r] * Sb[(size_t)r * dv + c];
            ob[c] = normalize ? s / den : s;
        }
        free(fq); free(fk);
    }
}

/* ---------------------------------------------------------------------------
 * Backward pass of the causal form (elu + 1, with the normaliser): given dO,
 * the gradients dq, dk, dv of L = sum_i dO_i . o_i.  The pages give no
 * gradient ("Linear Attention -- Math + Variants", Chunkwise parallelism:
 * training runs the parallel form); this is the chain rule applied to the
 * recurrence's definition, with n_i = phi(q_i)^T S_i, d_i = max(phi(q_i)^T z_i, eps),
 * o_i = n_i / d_i:
 *   dn_i = dO_i / d_i,  dd_i = -(dO_i . o_i) / d_i  (0 where the clamp binds),
 *   dphi(q_i) = S_i dn_i + dd_i z_i                    (S_i, z_i inclusive),
 *   dphi(k_j) = R_j v_j + r_j,  dv_j = R_j^T phi(k_j),
 *   R_j = sum_{i>=j} phi(q_i) dn_i^T,  r_j = sum_{i>=j} dd_i phi(q_i),
 *   dq = dphi(q) * phi'(q),  dk = dphi(k) * phi'(k),  phi'(x) = 1 (x > 0), exp(x).
 * Two passes per sequence: forward (S, z: o, d, dn, dd, dq) and backward (R, r:
 * dk, dv).  dO has the layout of v; dq, dk of q; dv of v (all double).
 * ------------------------------------------------------------------------- */
static double phi_prime(double x)
{
    return x > 0.0 ? 1.0 : exp(x);
}

void la_oracle_causal_backward(const void *q, const void *k, const void *v, const void *dout, int type,
                               double *dq, double *dk, double *dv, int BH, int N, int dkd, int dvd, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        const int64_t qb = (int64_t)bh * N * dkd, vb = (int64_t)bh * N * dvd;
        double *S = calloc((size_t)dkd * dvd, sizeof(double));
        double *z = calloc((size_t)dkd, sizeof(double));
        double *fq = malloc(sizeof(double) * dkd);
        double *fk = malloc(sizeof(double) * dkd);
        double *vt = malloc(sizeof(double) * dvd);
        double *dn = malloc(sizeof(double) * (size_t)N * dvd);  /* dn_i for the second pass */
        double *dd = malloc(sizeof(double) * (size_t)N);
        /* pass 1: t = 0 .. N-1 */
        for (int t = 0; t < N; ++t) {
            phi_row(q, type, qb, t, dkd, fq);
            phi_row(k, type, qb, t, dkd, fk);
            for (int c = 0; c < dvd; ++c)
                vt[c] = load(v, type, vb + (int64_t)t * dvd + c);
            for (int r = 0; r < dkd; ++r) {
                double *Sr = S + (size_t)r * dvd;
                for (int c = 0; c < dvd; ++c)
                    Sr[c] += fk[r] * vt[c];
                z[r] += fk[r];
            }
            double den = 0.0;
            for (int r = 0; r < dkd; ++r)
                den += fq[r] * z[r];
            const int clamped = !(den > eps);
            const double d = clamp_den(den, eps);
            double g = 0.0; /* dO_t . o_t */
            for (int c = 0; c < dvd; ++c) {
                double n = 0.0;
                for (int r = 0; r < dkd; ++r)
                    n += fq[r] * S[(size_t)r * dvd + c];
                const double go = load(dout, type, vb + (int64_t)t * dvd + c);
                g += go * (n / d);
                dn[(size_t)t * dvd + c] = go / d;
            }
            dd[t] = clamped ? 0.0 : -g / d;
            for (int r = 0; r < dkd; ++r) {
                double s = dd[t] * z[r];
                for (int c = 0; c < dvd; ++c)
                    s += S[(size_t)r * dvd + c] * dn[(size_t)t * dvd + c];
                dq[qb + (int64_t)t * dkd + r] = s * phi_prime(load(q, type, qb + (int64_t)t * dkd + r));
            }
        }
        /* pass 2: t = N-1 .. 0, R and r accumulate phi(q_i) dn_i^T and dd_i phi(q_i) for i >= t */
        double *R = S, *rr = z;
        memset(R, 0, sizeof(double) * (size_t)dkd * dvd);
        memset(rr, 0, sizeof(double) * (size_t)dkd);
        for (int t = N - 1; t >= 0; --t) {
            phi_row(q, type, qb, t, dkd, fq);
            phi_row(k, type, qb, t, dkd, fk);
            for (int r = 0; r < dkd; ++r) {
                double *Rr = R + (size_t)r * dvd;
                for (int c = 0; c < dvd; ++c)
                    Rr[c] += fq[r] * dn[(size_t)t * dvd + c];
                rr[r] += dd[t] * fq[r];
            }
            for (int r = 0; r < dkd; ++r) {
                double s = rr[r];
                for (int c = 0; c < dvd; ++c)
                    s += R[(size_t)r * dvd + c] * load(v, type, vb + (int64_t)t * dvd + c);
                dk[qb + (int64_t)t * dkd + r] = s * phi_prime(load(k, type, qb + (int64_t)t * dkd + r));
            }
            for (int c = 0; c < dvd; ++c) {
                double s = 0.0;
                for (int r = 0; r < dkd; ++r)
                    s += R[(size_t)r * dvd + c] * fk[r];
                dv[vb + (int64_t)t * dvd + c] = s;
            }
        }
        free(S); free(z); free(fq); free(fk); free(vt); free(dn); free(dd);
    }
}

/* ---------------------------------------------------------------------------
 * Performer FAVOR+ positive random features ("Linear Attention -- Math +
 * Variants", Performer: unbiased softmax by positive random features):
 *   phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m),  r = 0 .. m-1,
 * with E[phi(q) . phi(k)] = exp(q . k) for w_r ~ N(0, I).  x [rows, d] (any input
 * type), W [m, d] double (the random features are an input), out [rows, m] double.
 * ------------------------------------------------------------------------- */
void la_oracle_favor_features(const void *x, int type, const double *W, double *out, long long rows, int d, int m)
{
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < rows; ++i) {
        double nrm = 0.0;
        for (int c = 0; c < d; ++c) {
            const double xc = load(x, type, i * d + c);
            nrm += xc * xc;
        }
        for (int r = 0; r < m; ++r) {
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += W[(size_t)r * d + c] * load(x, type, i * d + c);
            out[i * m + r] = exp(dot - 0.5 * nrm) / sqrt((double)m);
        }
    }
}

/* Threads OpenMP will use (reported beside CPU timings). */
/* ---------------------------------------------------------------------------
 * Gated state, one gate per key feature ([wiki] "What is actually lost": gated
 * variants insert a decay, S_t = G_t (.) S_{t-1} + phi(k_t) v_t^T; [math] "RetNet
 * and gated linear attention": S_i = Diag(alpha_i) S_{i-1} + k_i v_i^T, the decay
 * computed from the token itself).
 * Readings: the gate values are an input, alpha [BH, N, dk] in [0, 1] (the
 * projection that makes them from the token is a trained layer, the caller's);
 * G_t = alpha_t 1^T, i.e. row r of S (key feature r) is scaled by alpha_t[r];
 * phi is applied to k as everywhere else; the normaliser z decays with the same
 * gate (the reading taken for the scalar decay above, which this reduces to when
 * every alpha_t[r] = gamma):
 *   S_t = Diag(alpha_t) S_{t-1} + phi(k_t) v_t^T,  z_t = alpha_t (.) z_{t-1} + phi(k_t),
 *   o_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps).
 * ------------------------------------------------------------------------- */
void la_oracle_causal_gated_recurrent(const void *q, const void *k, const void *v, int type,
                                      const double *alpha, double *o, int BH, int N, int dk,
                                      int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        double *S = calloc((size_t)dk * dv, sizeof(double));
        double *z = calloc((size_t)dk, sizeof(double));
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        double *vt = malloc(sizeof(double) * dv);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int t = 0; t < N; ++t) {
            phi_row(q, type, qb, t, dk, fq);
            phi_row(k, type, qb, t, dk, fk);
            const double *at = alpha + qb + (int64_t)t * dk;
            for (int c = 0; c < dv; ++c)
                vt[c] = load(v, type, vb + (int64_t)t * dv + c);
            /* S = Diag(alpha_t) S + phi(k_t) v_t^T ; z = alpha_t (.) z + phi(k_t) */
            for (int r = 0; r < dk; ++r) {
                double *Sr = S + (size_t)r * dv;
                for (int c = 0; c < dv; ++c)
                    Sr[c] = at[r] * Sr[c] + fk[r] * vt[c];
                z[r] = at[r] * z[r] + fk[r];
            }
            double den = 0.0;
            for (int r = 0; r < dk; ++r)
                den += fq[r] * z[r];
            double *ot = o + vb + (int64_t)t * dv;
            for (int c = 0; c < dv; ++c)
                ot[c] = 0.0;
            for (int r = 0; r < dk; ++r) {
                const double *Sr = S + (size_t)r * dv;
                for (int c = 0; c < dv; ++c)
                    ot[c] += fq[r] * Sr[c];
            }
            den = clamp_den(den, eps);
            for (int c = 0; c < dv; ++c)
                ot[c] /= den;
        }
        free(S); free(z); free(fq); free(fk); free(vt);
    }
}

/* The weighted pairwise form the gated recurrence unrolls to: key j reaches query
 * i >= j through feature r with weight prod_{s=j+1..i} alpha_s[r], so
 *   w_ij = sum_r phi(q_i)[r] phi(k_j)[r] prod_{s=j+1..i} alpha_s[r],
 *   o_i = sum_{j<=i} w_ij v_j / max(sum_{j<=i} w_ij, eps).
 * The products are built going back from j = i (empty product 1).  O(N^2 dk):
 * cross-check only. */
void la_oracle_causal_gated_quadratic(const void *q, const void *k, const void *v, int type,
                                      const double *alpha, double *o, int BH, int N, int dk,
                                      int dv, double eps)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < BH; ++bh) {
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        double *prod = malloc(sizeof(double) * dk);
        const int64_t qb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        for (int i = 0; i < N; ++i) {
            phi_row(q, type, qb, i, dk, fq);
            double *oi = o + vb + (int64_t)i * dv;
            for (int c = 0; c < dv; ++c)
                oi[c] = 0.0;
            for (int r = 0; r < dk; ++r)
                prod[r] = 1.0;
            double rowsum = 0.0;
            for (int j = i; j >= 0; --j) {
                if (j < i)
                    for (int r = 0; r < dk; ++r)
                        prod[r] *= alpha[qb + (int64_t)(j + 1) * dk + r];
                phi_row(k, type, qb, j, dk, fk);
                double w = 0.0;
                for (int r = 0; r < dk; ++r)
                    w += fq[r] * fk[r] * prod[r];
                rowsum += w;
                for (int c = 0; c < dv; ++c)
                    oi[c] += w * load(v, type, vb + (int64_t)j * dv + c);
            }
            rowsum = clamp_den(rowsum, eps);
            for (int c = 0; c < dv; ++c)
                oi[c] /= rowsum;
        }
        free(fq); free(fk); free(prod);
    }
}

/* One gated decode step, state in place: S = Diag(alpha) S + phi(k) v^T,
 * z = alpha (.) z + phi(k), then o = phi(q)^T S / max(phi(q)^T z, eps).
 * alpha [BH, dk]. */
void la_oracle_decode_step_gated(double *S, double *z, const void *q, const void *k,
                                 const void *v, int type, const double *alpha, double *o, int BH,
                                 int dk, int dv, double eps)
{
#pragma omp parallel for schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * dk * dv;
        double *zb = z + (size_t)bh * dk;
        double *ob = o + (size_t)bh * dv;
        const double *ab = alpha + (size_t)bh * dk;
        double *fq = malloc(sizeof(double) * dk);
        double *fk = malloc(sizeof(double) * dk);
        for (int r = 0; r < dk; ++r) {
            fq[r] = la_oracle_phi(load(q, type, (int64_t)bh * dk + r));
            fk[r] = la_oracle_phi(load(k, type, (int64_t)bh * dk + r));
        }
        for (int r = 0; r < dk; ++r) {
            for (int c = 0; c < dv; ++c)
                Sb[(size_t)r * dv + c] = ab[r] * Sb[(size_t)r * dv + c] + fk[r] * load(v, type, (int64_t)bh * dv + c);
            zb[r] = ab[r] * zb[r] + fk[r];
        }
        double den = 0.0;
        for (int r = 0; r < dk; ++r)
            den += fq[r] * zb[r];
        den = clamp_den(den, eps);
        for (int c = 0; c < dv; ++c) {
            double s = 0.0;
            for (int r = 0; r < dk; ++r)
                s += fq[r] * Sb[(size_t)r * dv + c];
            ob[c] = s / den;
        }
        free(fq); free(fk);
    }
}

/* State after N tokens of the gated recurrence from a zero state (a prefill):
 * S = sum_t Diag(prod_{s=t+1..N-1} alpha_s) phi(k_t) v_t^T, z likewise, written as
 * the recurrence itself.  S [BH, dk, dv] and z [BH, dk] are overwritten. */
void la_oracle_prefill_state_gated(const void *k, const void *v, int type, const double *alpha,
                                   double *S, double *z, int BH, int N, int dk, int dv)
{
#pragma omp parallel for schedule(static)
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * dk * dv;
        double *zb = z + (size_t)bh * dk;
        double *fk = malloc(sizeof(double) * dk);
        const int64_t kb = (int64_t)bh * N * dk, vb = (int64_t)bh * N * dv;
        memset(Sb, 0, sizeof(double) * dk * dv);
        memset(zb, 0, sizeof(double) * dk);
        for (int t = 0; t < N; ++t) {
            phi_row(k, type, kb, t, dk, fk);
            const double *at = alpha + kb + (int64_t)t * dk;
            for (int r = 0; r < dk; ++r) {
                for (int c = 0; c < dv; ++c)
                    Sb[(size_t)r * dv + c] = at[r] * Sb[(size_t)r * dv + c] + fk[r] * load(v, type, vb + (int64_t)t * dv + c);
                zb[r] = at[r] * zb[r] + fk[r];
            }
        }
        free(fk);
    }
}

int la_oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
