// Gated state with one gate per key feature ("Linear Attention",
// aiwiki.thehackersbrain.dev, What is actually lost: gated variants insert a
// decay, S_t = G_t (.) S_{t-1} + phi(k_t) v_t^T; "Linear Attention -- Math +
// Variants", aicassindra.com, RetNet and gated linear attention:
// S_i = Diag(alpha_i) S_{i-1} + k_i v_i^T with the decay computed from the token):
//
//   S_t = Diag(alpha_t) S_{t-1} + phi(k_t) v_t^T,   z_t = alpha_t (.) z_{t-1} + phi(k_t),
//   o_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps)
//
// with the gate alpha [B, H, N, dk] (fp32, in [0, 1]) given by the caller.
//
// CUDA cores, fp32.  Column c of S evolves on its own (row r is scaled by
// alpha_t[r] and takes phi(k_t)[r] v_t[c]), so the recurrence is split over value
// columns: a CTA of 4 warps owns 32 columns of one head; in a warp, lane
// (rq, c) = (lane / 8, lane % 8) holds rows [rq dk/4, (rq+1) dk/4) of column
// 8 w + c of S and the same rows of z (the z rows are repeated across the
// column lanes: each computes the denominator it needs).  Per token a lane
// updates its rows, forms its partial phi(q).S and phi(q).z, and two shuffles
// add the four row quarters.  The tokens stream through shared memory in chunks
// of 32: the next chunk's q, k, alpha and v are copied asynchronously (cp.async)
// while the current chunk runs, then phi is applied once per chunk.
//
// The decode step is the recurrence's body for one token over all heads (the
// state streams through once, as in the ungated step); the prefix state is the
// recurrence without outputs.
#include <cuda_pipeline.h>

#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kT = 32;        // tokens per chunk
constexpr int kGThreads = 128;
constexpr int kCols = 32;     // value columns per CTA

template <typename T, int DK>
struct GSmem {
    // raw inputs of the chunk in flight (async copies), then the chunk in use
    T rq[kT][DK], rk[kT][DK];
    float ra[kT][DK], rv[kT][kCols];
    float fq[kT][DK], fk[kT][DK], al[kT][DK], v[kT][kCols];
    float out[kT][kCols];
};

// Async copies of one chunk (tokens [t0, t0 + n)) into the raw buffers; 4-byte
// granules so that any dv and column offset are covered, 16-byte granules where
// rows are whole.
template <typename T, int DK, bool kState>
__device__ __forceinline__ void issue_chunk(GSmem<T, DK> &sm, const T *q, const T *k, const float *alpha,
                                            const T *v, int t0, int n, int dv, int col0, int tid)
{
    constexpr int kElemPer16 = 16 / sizeof(T);
    for (int x = tid; x < n * (DK / kElemPer16); x += kGThreads) {
        const int t = x / (DK / kElemPer16), e = (x % (DK / kElemPer16)) * kElemPer16;
        if (!kState) __pipeline_memcpy_async(&sm.rq[t][e], q + (size_t)(t0 + t) * DK + e, 16);
        __pipeline_memcpy_async(&sm.rk[t][e], k + (size_t)(t0 + t) * DK + e, 16);
    }
    for (int x = tid; x < n * (DK / 4); x += kGThreads) {
        const int t = x / (DK / 4), e = (x % (DK / 4)) * 4;
        __pipeline_memcpy_async(&sm.ra[t][e], alpha + (size_t)(t0 + t) * DK + e, 16);
    }
    const int ncol = min(kCols, dv - col0);
    for (int x = tid; x < n * kCols; x += kGThreads) {
        const int t = x / kCols, c = x % kCols;
        if (c < ncol) {
            if constexpr (sizeof(T) == 4)
                __pipeline_memcpy_async(&sm.rv[t][c], v + (size_t)(t0 + t) * dv + col0 + c, 4);
            else
                sm.rv[t][c] = Elem<T>::to_f32(v[(size_t)(t0 + t) * dv + col0 + c]);
        }
    }
    __pipeline_commit();
}

// Grid (BH, ceil(dv / 32)).  kState: no outputs; the final S (rows x this CTA's
// columns) and z are written to S_out, z_out.
template <typename T, int DK, bool kState>
__global__ void __launch_bounds__(kGThreads)
gated_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
             const float *__restrict__ alpha, T *__restrict__ o, float *__restrict__ S_out,
             float *__restrict__ z_out, int N, int dv, float eps)
{
    constexpr int kRpl = DK / 4;  // rows per lane
    extern __shared__ __align__(16) uint8_t gsm_raw[];
    GSmem<T, DK> &sm = *reinterpret_cast<GSmem<T, DK> *>(gsm_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rq = lane >> 3, cl = lane & 7;
    const int col = warp * 8 + cl;            // column within the CTA's 32
    const int col0 = blockIdx.y * kCols;
    const size_t bh = blockIdx.x;
    const T *qh = q + bh * N * DK, *kh = k + bh * N * DK, *vh = v + bh * N * dv;
    const float *ah = alpha + bh * N * DK;
    const bool col_ok = col0 + col < dv;

    float s[kRpl], z[kRpl];
#pragma unroll
    for (int i = 0; i < kRpl; ++i) s[i] = z[i] = 0.f;

    const int n_chunks = (N + kT - 1) / kT;
    if (n_chunks > 0) issue_chunk<T, DK, kState>(sm, qh, kh, ah, vh, 0, min(kT, N), dv, col0, tid);
    for (int j = 0; j < n_chunks; ++j) {
        const int t0 = j * kT, n = min(kT, N - t0);
        // the chunk's raw inputs have landed: phi once, into the buffers in use
        __pipeline_wait_prior(0);
        __syncthreads();
        for (int x = tid; x < n * DK; x += kGThreads) {
            const int t = x / DK, e = x % DK;
            if (!kState) sm.fq[t][e] = Elem<T>::phi(Elem<T>::to_f32(sm.rq[t][e]));
            sm.fk[t][e] = Elem<T>::phi(Elem<T>::to_f32(sm.rk[t][e]));
            sm.al[t][e] = sm.ra[t][e];
        }
        for (int x = tid; x < n * kCols; x += kGThreads) sm.v[x / kCols][x % kCols] = sm.rv[x / kCols][x % kCols];
        __syncthreads();
        // the next chunk's copies run while this one is computed
        if (j + 1 < n_chunks) issue_chunk<T, DK, kState>(sm, qh, kh, ah, vh, t0 + kT, min(kT, N - t0 - kT), dv, col0, tid);
        for (int t = 0; t < n; ++t) {
            const float vc = sm.v[t][col];
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int i4 = 0; i4 < kRpl; i4 += 4) {
                const float4 a = *reinterpret_cast<const float4 *>(&sm.al[t][rq * kRpl + i4]);
                const float4 b = *reinterpret_cast<const float4 *>(&sm.fk[t][rq * kRpl + i4]);
                const float aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    s[i4 + u] = fmaf(aa[u], s[i4 + u], bb[u] * vc);
                    z[i4 + u] = fmaf(aa[u], z[i4 + u], bb[u]);
                }
                if (!kState) {
                    const float4 c = *reinterpret_cast<const float4 *>(&sm.fq[t][rq * kRpl + i4]);
                    const float cc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        num = fmaf(cc[u], s[i4 + u], num);
                        den = fmaf(cc[u], z[i4 + u], den);
                    }
                }
            }
            if (!kState) {
                num += __shfl_xor_sync(0xffffffffu, num, 8);
                den += __shfl_xor_sync(0xffffffffu, den, 8);
                num += __shfl_xor_sync(0xffffffffu, num, 16);
                den += __shfl_xor_sync(0xffffffffu, den, 16);
                if (rq == 0) sm.out[t][col] = num / fmaxf(den, eps);
            }
        }
        if (!kState) {
            __syncthreads();
            const int ncol = min(kCols, dv - col0);
            for (int x = tid; x < n * kCols; x += kGThreads) {
                const int t = x / kCols, c = x % kCols;
                if (c < ncol) o[(bh * N + t0 + t) * dv + col0 + c] = Elem<T>::from_f32(sm.out[t][c]);
            }
        }
    }
    if (kState) {
        if (col_ok) {
#pragma unroll
            for (int i = 0; i < kRpl; ++i) S_out[(bh * DK + rq * kRpl + i) * dv + col0 + col] = s[i];
        }
        if (blockIdx.y == 0 && warp == 0 && cl == 0) {
#pragma unroll
            for (int i = 0; i < kRpl; ++i) z_out[bh * DK + rq * kRpl + i] = z[i];
        }
    }
}

// One gated decode step, one CTA per head: S = Diag(alpha) S + phi(k) v^T,
// z = alpha (.) z + phi(k), o = phi(q)^T S / max(phi(q)^T z, eps).  Each thread owns
// float4 column groups of a few rows; all state loads are issued before any
// arithmetic; partial numerators are reduced over row groups in shared memory.
constexpr int kDThreads = 256;

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kDThreads)
gated_decode_kernel(float *__restrict__ S, float *__restrict__ z, const T *__restrict__ q,
                    const T *__restrict__ k, const T *__restrict__ v, T *__restrict__ o,
                    const float *__restrict__ alpha, float eps)
{
    constexpr int kCols4 = DV / 4, kRowGroups = kDThreads / kCols4, kRows = DK / kRowGroups;
    static_assert(kRows >= 1 && DK % kRowGroups == 0, "shape");
    __shared__ float fq[DK], fk[DK], al[DK];
    __shared__ float4 part[kRowGroups][kCols4];
    __shared__ float red[kDThreads / 32];
    const size_t head = blockIdx.x;
    const int tid = threadIdx.x, cg = tid % kCols4, rg = tid / kCols4;
    float4 *Sh = reinterpret_cast<float4 *>(S + head * DK * DV);
    float4 s[kRows];
#pragma unroll
    for (int m = 0; m < kRows; ++m) s[m] = __ldcs(Sh + (size_t)(rg + m * kRowGroups) * kCols4 + cg);
    for (int r = tid; r < DK; r += kDThreads) {
        fq[r] = Elem<T>::phi(Elem<T>::to_f32(q[head * DK + r]));
        fk[r] = Elem<T>::phi(Elem<T>::to_f32(k[head * DK + r]));
        al[r] = alpha[head * DK + r];
    }
    float vc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) vc[u] = Elem<T>::to_f32(v[head * DV + 4 * cg + u]);
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
        const int r = rg + m * kRowGroups;
        const float a = al[r], b = fk[r], c = fq[r];
        float4 x = s[m];
        x.x = fmaf(a, x.x, b * vc[0]); x.y = fmaf(a, x.y, b * vc[1]);
        x.z = fmaf(a, x.z, b * vc[2]); x.w = fmaf(a, x.w, b * vc[3]);
        __stcs(Sh + (size_t)r * kCols4 + cg, x);
        acc.x += c * x.x; acc.y += c * x.y; acc.z += c * x.z; acc.w += c * x.w;
    }
    part[rg][cg] = acc;
    float d = 0.f;
    for (int r = tid; r < DK; r += kDThreads) {
        const float zn = fmaf(al[r], z[head * DK + r], fk[r]);
        z[head * DK + r] = zn;
        d += fq[r] * zn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if ((tid & 31) == 0) red[tid >> 5] = d;
    __syncthreads();
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kDThreads / 32; ++w) den += red[w];
    const float inv = 1.f / fmaxf(den, eps);
    if (tid < DV) {
        const int c4 = tid >> 2, l4 = tid & 3;
        float num = 0.f;
#pragma unroll 8
        for (int g = 0; g < kRowGroups; ++g) {
            const float4 p = part[g][c4];
            num += l4 == 0 ? p.x : l4 == 1 ? p.y : l4 == 2 ? p.z : p.w;
        }
        o[head * DV + tid] = Elem<T>::from_f32(num * inv);
    }
}

template <typename T, int DK, bool kState>
la_status launch_gated(const void *q, const void *k, const void *v, const float *alpha, void *o, float *S,
                       float *z, int BH, int N, int dv, float eps, cudaStream_t stream)
{
    auto kern = gated_kernel<T, DK, kState>;
    const int smem = (int)sizeof(GSmem<T, DK>);
    la_status st = ensure_smem((const void *)kern, smem);
    if (st != LA_OK) return st;
    dim3 grid(BH, ceil_div(dv, kCols));
    count_launches();
    kern<<<grid, kGThreads, smem, stream>>>((const T *)q, (const T *)k, (const T *)v, alpha, (T *)o, S, z, N, dv, eps);
    return cuda_status(cudaGetLastError());
}

template <typename T, bool kState>
la_status gated_by_dk(const void *q, const void *k, const void *v, const float *alpha, void *o, float *S, float *z,
                      int BH, int N, int dk, int dv, float eps, cudaStream_t stream)
{
    switch (dk) {
    case 32: return launch_gated<T, 32, kState>(q, k, v, alpha, o, S, z, BH, N, dv, eps, stream);
    case 64: return launch_gated<T, 64, kState>(q, k, v, alpha, o, S, z, BH, N, dv, eps, stream);
    case 128: return launch_gated<T, 128, kState>(q, k, v, alpha, o, S, z, BH, N, dv, eps, stream);
    }
    return LA_ERR_UNSUPPORTED;
}

template <typename T, int DK>
la_status decode_by_dv(float *S, float *z, const void *q, const void *k, const void *v, void *o, const float *alpha,
                       int BH, int dv, float eps, cudaStream_t stream)
{
    count_launches();
    switch (dv) {
    case 32:
        gated_decode_kernel<T, DK, 32><<<BH, kDThreads, 0, stream>>>(S, z, (const T *)q, (const T *)k, (const T *)v,
                                                                     (T *)o, alpha, eps);
        break;
    case 64:
        gated_decode_kernel<T, DK, 64><<<BH, kDThreads, 0, stream>>>(S, z, (const T *)q, (const T *)k, (const T *)v,
                                                                     (T *)o, alpha, eps);
        break;
    case 128:
        gated_decode_kernel<T, DK, 128><<<BH, kDThreads, 0, stream>>>(S, z, (const T *)q, (const T *)k, (const T *)v,
                                                                      (T *)o, alpha, eps);
        break;
    default: return LA_ERR_UNSUPPORTED;
    }
    return cuda_status(cudaGetLastError());
}

template <typename T>
la_status decode_by_dk(float *S, float *z, const void *q, const void *k, const void *v, void *o, const float *alpha,
                       int BH, int dk, int dv, float eps, cudaStream_t stream)
{
    switch (dk) {
    case 32: return decode_by_dv<T, 32>(S, z, q, k, v, o, alpha, BH, dv, eps, stream);
    case 64: return decode_by_dv<T, 64>(S, z, q, k, v, o, alpha, BH, dv, eps, stream);
    case 128: return decode_by_dv<T, 128>(S, z, q, k, v, o, alpha, BH, dv, eps, stream);
    }
    return LA_ERR_UNSUPPORTED;
}

}  // namespace

la_status causal_gated(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH, int N,
                       int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream)
{
    // the chunked form (la_gated_chunk.cu); the token-by-token recurrence below serves
    // the prefix state and stays available as a reference for it
    return causal_gated_chunked(q, k, v, alpha, o, BH, N, dk, dv, eps, dtype, stream);
}

la_status causal_gated_recurrent(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH,
                                 int N, int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream)
{
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    return dtype == LA_F32 ? gated_by_dk<float, false>(q, k, v, alpha, o, nullptr, nullptr, BH, N, dk, dv, eps, stream)
                           : gated_by_dk<__nv_bfloat16, false>(q, k, v, alpha, o, nullptr, nullptr, BH, N, dk, dv, eps,
                                                              stream);
}

la_status state_gated(const void *k, const void *v, const float *alpha, float *S, float *z, int BH, int N, int dk,
                      int dv, la_dtype dtype, cudaStream_t stream)
{
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    return dtype == LA_F32 ? gated_by_dk<float, true>(k, k, v, alpha, nullptr, S, z, BH, N, dk, dv, 0.f, stream)
                           : gated_by_dk<__nv_bfloat16, true>(k, k, v, alpha, nullptr, S, z, BH, N, dk, dv, 0.f, stream);
}

la_status decode_step_gated(float *S, float *z, const void *q, const void *k, const void *v, void *o,
                            const float *alpha, int BH, int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream)
{
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    return dtype == LA_F32 ? decode_by_dk<float>(S, z, q, k, v, o, alpha, BH, dk, dv, eps, stream)
                           : decode_by_dk<__nv_bfloat16>(S, z, q, k, v, o, alpha, BH, dk, dv, eps, stream);
}

}  // namespace la
