// Causal forward with the gated state (one gate per key feature) in chunks, on the
// CUDA cores in fp32: the same recurrence as la_gated.cu ("Linear Attention",
// aiwiki.thehackersbrain.dev, What is actually lost; "Linear Attention -- Math +
// Variants", aicassindra.com, RetNet and gated linear attention)
//
//   S_t = Diag(alpha_t) S_{t-1} + phi(k_t) v_t^T,   z_t = alpha_t (.) z_{t-1} + phi(k_t),
//   o_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps),
//
// written over chunks of C tokens ([wiki] listing linear_attention_chunked for the
// ungated case; [math] Chunkwise parallelism).  Inside a chunk, with
// D_f(t, s) = prod_{s < u <= t} alpha_u[f] and Lambda_t[f] = prod_{u <= t} alpha_u[f]:
//
//   phi(q_t)^T S_t = sum_f phi(q_t)[f] Lambda_t[f] S_in[f, :]                 (state before the chunk)
//                  + sum_{s <= t} A(t, s) v_s,   A(t, s) = sum_f phi(q_t)[f] phi(k_s)[f] D_f(t, s)
//
// and the chunk's own contribution to the state after it is
// sum_s Diag(D_f(C-1, s)) phi(k_s) v_s^T, the state carried across by Lambda_{C-1}.
// Every decay is a running product of gates, never a quotient of products, so gates
// of exactly 0 (and products that underflow) stay exact.  Three launches:
//
//   1. chunk states   dS_c = W^T V, dz_c = W^T 1 with W[s] = phi(k_s) (.) prod_{u > s} alpha_u,
//                     lam_c = prod_s alpha_s
//   2. scan           [S | z] before chunk c: S_in(c + 1) = lam_c (.) S_in(c) + dS_c (rows scaled)
//   3. outputs        A(t, s) by a running product per key (w <- w (.) alpha_t, A = phi(q_t).w),
//                     o_t = ([A | qt] [V ; S_in])_t / max(sum_s A(t, s) + qt_t . z_in, eps),
//                     qt_t = phi(q_t) (.) Lambda_t.
// The two products are register-tiled (each thread a small block of outputs, operand
// vectors read from shared memory as float2 / float4).
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kCh = 32;       // tokens per chunk
constexpr int kThr = 256;     // threads per CTA

// Rows [0, len) of a contiguous [rows x W] block into shared memory as fp32 ([kCh][LD]);
// rows at or past len read as `fill`; f is applied to the live values.  The block is
// 16-byte aligned (rows of W elements from a 16-byte aligned tensor, W a multiple of
// 32): every 16-byte load of a thread is issued before any is converted.
template <typename T, int W, int LD, typename F>
__device__ __forceinline__ void load_rows_f32(float *dst, const T *src, int len, float fill, F f, int tid)
{
    constexpr int V = 16 / (int)sizeof(T);  // elements per 16-byte vector
    constexpr int NV = kCh * W / V;
    constexpr int PER = (NV + kThr - 1) / kThr;
    static_assert(W % V == 0, "rows are whole vectors");
    uint4 buf[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = tid + i * kThr;
        if (e < NV && (e * V) / W < len) buf[i] = __ldg(reinterpret_cast<const uint4 *>(src) + e);
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = tid + i * kThr;
        if (e < NV) {
            const int r = (e * V) / W, c = (e * V) % W;
            const T *x = reinterpret_cast<const T *>(&buf[i]);
#pragma unroll
            for (int j = 0; j < V; ++j) dst[r * LD + c + j] = r < len ? f(Elem<T>::to_f32(x[j])) : fill;
        }
    }
}

// Slot of a chunk (fp32): S [DK][DV], then z [DK], then the chunk's gate product lam [DK].
template <int DK, int DV>
struct Slot {
    static constexpr int kZ = DK * DV;
    static constexpr int kLam = kZ + DK;
    static constexpr int kAll = kLam + DK;
};

// ---------------------------------------------------------------------- 1. chunk states
template <int DK, int DV>
struct StateSmem {
    float w[kCh][DK];   // phi(k_s), then W[s] = phi(k_s) (.) prod_{u > s} alpha_u
    float al[kCh][DK];
    float v[kCh][DV];
};

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr)
gated_chunk_state(const T *__restrict__ k, const T *__restrict__ v, const float *__restrict__ alpha,
                  float *__restrict__ slots, int N, int nC)
{
    extern __shared__ __align__(16) float smf[];
    StateSmem<DK, DV> &sm = *reinterpret_cast<StateSmem<DK, DV> *>(smf);
    const int c = blockIdx.x % nC, bh = blockIdx.x / nC, tid = threadIdx.x;
    const int t0 = c * kCh, len = min(kCh, N - t0);
    const size_t rk = ((size_t)bh * N + t0) * DK, rv = ((size_t)bh * N + t0) * DV;
    load_rows_f32<T, DK, DK>(&sm.w[0][0], k + rk, len, 0.f, [](float x) { return Elem<T>::phi(x); }, tid);
    load_rows_f32<float, DK, DK>(&sm.al[0][0], alpha + rk, len, 1.f, [](float x) { return x; }, tid);
    load_rows_f32<T, DV, DV>(&sm.v[0][0], v + rv, len, 0.f, [](float x) { return x; }, tid);
    __syncthreads();
    float *slot = slots + ((size_t)bh * nC + c) * Slot<DK, DV>::kAll;
    if (tid < DK) {  // suffix gate products, in place; the whole chunk's product to lam
        float p = 1.f;
        for (int s = kCh - 1; s >= 0; --s) {
            sm.w[s][tid] *= p;
            p *= sm.al[s][tid];
        }
        slot[Slot<DK, DV>::kLam + tid] = p;
    }
    __syncthreads();
    // dS = W^T V: thread tile FR x 4 (features x columns); DK / FR x DV / 4 = 256 threads
    constexpr int CG = DV / 4, FR = DK * DV / (kThr * 4);
    static_assert(FR >= 1 && (DK / FR) * CG == kThr, "tile shape");
    const int cg = tid % CG, fg = tid / CG, f0 = fg * FR, c0 = cg * 4;
    float acc[FR][4], zacc[FR];
#pragma unroll
    for (int a = 0; a < FR; ++a) {
        zacc[a] = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
    }
#pragma unroll 4
    for (int s = 0; s < kCh; ++s) {
        const float4 vv = *reinterpret_cast<const float4 *>(&sm.v[s][c0]);
#pragma unroll
        for (int a = 0; a < FR; ++a) {
            const float wv = sm.w[s][f0 + a];
            acc[a][0] += wv * vv.x; acc[a][1] += wv * vv.y; acc[a][2] += wv * vv.z; acc[a][3] += wv * vv.w;
            zacc[a] += wv;
        }
    }
#pragma unroll
    for (int a = 0; a < FR; ++a) {
        *reinterpret_cast<float4 *>(slot + (f0 + a) * DV + c0) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        if (cg == 0) slot[Slot<DK, DV>::kZ + f0 + a] = zacc[a];
    }
}

// ---------------------------------------------------------------------- 2. scan
// Thread = (head, float4 of S or z); S_in(0) = 0, S_in(c + 1) = lam_c (.) S_in(c) + dS_c
// (rows scaled by the chunk's gate product), written in place of dS_c.  Eight chunks'
// loads in flight before their stores.
template <int DK, int DV>
__global__ void __launch_bounds__(kThr)
gated_chunk_scan(float *__restrict__ slots, int nC, long long total4)
{
    constexpr int E4 = (DK * DV + DK) / 4;
    const long long g = (long long)blockIdx.x * kThr + threadIdx.x;
    if (g >= total4) return;
    const long long bh = g / E4;
    const int e = (int)(g % E4) * 4;
    const bool in_s = e < Slot<DK, DV>::kZ;
    // the gate row of these four elements: one feature for S (DV is a multiple of 4),
    // four consecutive features for z
    const int lam_off = in_s ? Slot<DK, DV>::kLam + e / DV : Slot<DK, DV>::kLam + (e - Slot<DK, DV>::kZ);
    float *p = slots + bh * (long long)nC * Slot<DK, DV>::kAll;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < nC; i += 8) {
        float4 x[8], lam[8];
        const int m = min(8, nC - i);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (u < m) {
                const float *sl = p + (long long)(i + u) * Slot<DK, DV>::kAll;
                x[u] = __ldcg(reinterpret_cast<const float4 *>(sl + e));
                if (in_s) {
                    const float l = __ldcg(sl + lam_off);
                    lam[u] = make_float4(l, l, l, l);
                } else {
                    lam[u] = __ldcg(reinterpret_cast<const float4 *>(sl + lam_off));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (u < m) {
                __stcg(reinterpret_cast<float4 *>(p + (long long)(i + u) * Slot<DK, DV>::kAll + e), run);
                run.x = lam[u].x * run.x + x[u].x;
                run.y = lam[u].y * run.y + x[u].y;
                run.z = lam[u].z * run.z + x[u].z;
                run.w = lam[u].w * run.w + x[u].w;
            }
        }
    }
}

// ---------------------------------------------------------------------- 3. outputs
// The left factor of the output product, [A | qt] ([kCh rows] x [kCh + DK]), is kept
// transposed (LT[k][t]) so that a thread's two rows are one float2; the right factor
// [V ; S_in] ([kCh + DK] x DV) row-major.
template <int DK, int DV>
struct OutSmem {
    float fq[kCh][DK], fk[kCh][DK], al[kCh][DK];
    float lt[kCh + DK][kCh];   // [A | qt] transposed
    float rb[kCh + DK][DV];    // [V ; S_in]
    float zin[DK];
    float den[kCh];
};

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThr)
gated_chunk_out(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                const float *__restrict__ alpha, const float *__restrict__ slots, T *__restrict__ o, int N, int nC,
                float eps)
{
    extern __shared__ __align__(16) float smf[];
    OutSmem<DK, DV> &sm = *reinterpret_cast<OutSmem<DK, DV> *>(smf);
    const int c = blockIdx.x % nC, bh = blockIdx.x / nC, tid = threadIdx.x;
    const int t0 = c * kCh, len = min(kCh, N - t0);
    const size_t rk = ((size_t)bh * N + t0) * DK, rv = ((size_t)bh * N + t0) * DV;
    auto phi = [](float x) { return Elem<T>::phi(x); };
    load_rows_f32<T, DK, DK>(&sm.fq[0][0], q + rk, len, 0.f, phi, tid);
    load_rows_f32<T, DK, DK>(&sm.fk[0][0], k + rk, len, 0.f, phi, tid);
    load_rows_f32<float, DK, DK>(&sm.al[0][0], alpha + rk, len, 1.f, [](float x) { return x; }, tid);
    load_rows_f32<T, DV, DV>(&sm.rb[0][0], v + rv, len, 0.f, [](float x) { return x; }, tid);
    {
        const float *slot = slots + ((size_t)bh * nC + c) * Slot<DK, DV>::kAll;
        const float4 *s4 = reinterpret_cast<const float4 *>(slot);
        for (int e = tid; e < DK * DV / 4; e += kThr)
            *reinterpret_cast<float4 *>(&sm.rb[kCh][0] + 4 * e) = __ldcg(s4 + e);
        if (tid < DK) sm.zin[tid] = __ldcg(slot + Slot<DK, DV>::kZ + tid);
    }
    __syncthreads();
    // qt = phi(q) (.) Lambda (the running gate product from the chunk's start), transposed
    if (tid < DK) {
        float p = 1.f;
        for (int t = 0; t < kCh; ++t) {
            p *= sm.al[t][tid];
            sm.lt[kCh + tid][t] = sm.fq[t][tid] * p;
        }
    }
    // A(t, s): thread (s, g) carries w = phi(k_s) (.) prod_{s < u <= t} alpha_u over the
    // features [g F, (g + 1) F) and adds phi(q_t) . w; the eight feature groups of one s
    // are adjacent lanes and sum by shuffles
    {
        constexpr int G = 8, F = DK / G;
        const int s = tid / G, g = tid % G, f0 = g * F;
        float w[F];
#pragma unroll
        for (int j = 0; j < F; ++j) w[j] = sm.fk[s][f0 + j];
        const int s_lo = (tid / 32) * (32 / G);  // the smallest s of this warp
        for (int t = s_lo; t < kCh; ++t) {
            const bool live = t >= s;
            float part = 0.f;
            if (live) {
                if (t > s) {
#pragma unroll
                    for (int j = 0; j < F; ++j) w[j] *= sm.al[t][f0 + j];
                }
#pragma unroll
                for (int j = 0; j < F; ++j) part += sm.fq[t][f0 + j] * w[j];
            }
#pragma unroll
            for (int off = 1; off < G; off <<= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if (g == 0 && live) sm.lt[s][t] = part;
        }
        if (g == 0)
            for (int t = 0; t < s; ++t) sm.lt[s][t] = 0.f;  // above the diagonal
    }
    __syncthreads();
    if (tid < kCh) {  // den_t = sum_s A(t, s) + qt_t . z_in
        float d = 0.f;
        for (int s = 0; s < kCh; ++s) d += sm.lt[s][tid];
#pragma unroll 8
        for (int f = 0; f < DK; ++f) d += sm.lt[kCh + f][tid] * sm.zin[f];
        sm.den[tid] = d;
    }
    __syncthreads();
    // O = [A | qt] [V ; S_in]: thread tile 2 rows x CT columns (16 row pairs x 16 column groups)
    constexpr int CT = DV / 16;
    const int rp = tid / 16, cgp = tid % 16, r0 = 2 * rp, c0 = cgp * CT;
    float acc[2][CT];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < CT; ++b) acc[a][b] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < kCh + DK; ++kk) {
        const float2 l2 = *reinterpret_cast<const float2 *>(&sm.lt[kk][r0]);
        float bv[CT];
        if constexpr (CT % 4 == 0) {
#pragma unroll
            for (int b = 0; b < CT; b += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(&sm.rb[kk][c0 + b]);
                bv[b] = x.x; bv[b + 1] = x.y; bv[b + 2] = x.z; bv[b + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int b = 0; b < CT; b += 2) {
                const float2 x = *reinterpret_cast<const float2 *>(&sm.rb[kk][c0 + b]);
                bv[b] = x.x; bv[b + 1] = x.y;
            }
        }
#pragma unroll
        for (int b = 0; b < CT; ++b) {
            acc[0][b] += l2.x * bv[b];
            acc[1][b] += l2.y * bv[b];
        }
    }
#pragma unroll
    for (int a = 0; a < 2; ++a) {
        const int t = r0 + a;
        if (t < len) {
            const float inv = 1.f / fmaxf(sm.den[t], eps);
            T *orow = o + rv + (size_t)t * DV + c0;
#pragma unroll
            for (int b = 0; b < CT; ++b) orow[b] = Elem<T>::from_f32(acc[a][b] * inv);
        }
    }
}

template <typename T, int DK, int DV>
la_status launch(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH, int N, float eps,
                 cudaStream_t stream)
{
    const int nC = ceil_div(N, kCh);
    const size_t floats = (size_t)BH * nC * Slot<DK, DV>::kAll;
    Scratch scratch;
    void *base = nullptr;
    la_status st = data_workspace(stream, sizeof(float) * floats, &base);
    if (st != LA_OK) {
        st = scratch.alloc(sizeof(float) * floats, stream);
        if (st != LA_OK) return st;
        base = scratch.ptr;
    }
    float *slots = (float *)base;
    const int ssmem = (int)sizeof(StateSmem<DK, DV>), osmem = (int)sizeof(OutSmem<DK, DV>);
    st = ensure_smem((const void *)gated_chunk_state<T, DK, DV>, ssmem);
    if (st == LA_OK) st = ensure_smem((const void *)gated_chunk_out<T, DK, DV>, osmem);
    if (st != LA_OK) return st;
    const unsigned grid = (unsigned)(BH * nC);
    const long long total4 = (long long)BH * ((DK * DV + DK) / 4);
    count_launches(3);
    gated_chunk_state<T, DK, DV><<<grid, kThr, ssmem, stream>>>((const T *)k, (const T *)v, alpha, slots, N, nC);
    gated_chunk_scan<DK, DV><<<(unsigned)((total4 + kThr - 1) / kThr), kThr, 0, stream>>>(slots, nC, total4);
    gated_chunk_out<T, DK, DV><<<grid, kThr, osmem, stream>>>((const T *)q, (const T *)k, (const T *)v, alpha, slots,
                                                              (T *)o, N, nC, eps);
    return cuda_status(cudaGetLastError());
}

template <typename T, int DK>
la_status by_dv(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH, int N, int dv,
                float eps, cudaStream_t stream)
{
    switch (dv) {
    case 32: return launch<T, DK, 32>(q, k, v, alpha, o, BH, N, eps, stream);
    case 64: return launch<T, DK, 64>(q, k, v, alpha, o, BH, N, eps, stream);
    case 128: return launch<T, DK, 128>(q, k, v, alpha, o, BH, N, eps, stream);
    }
    return LA_ERR_UNSUPPORTED;
}

template <typename T>
la_status by_dk(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH, int N, int dk,
                int dv, float eps, cudaStream_t stream)
{
    switch (dk) {
    case 32: return by_dv<T, 32>(q, k, v, alpha, o, BH, N, dv, eps, stream);
    case 64: return by_dv<T, 64>(q, k, v, alpha, o, BH, N, dv, eps, stream);
    case 128: return by_dv<T, 128>(q, k, v, alpha, o, BH, N, dv, eps, stream);
    }
    return LA_ERR_UNSUPPORTED;
}

}  // namespace

la_status causal_gated_chunked(const void *q, const void *k, const void *v, const float *alpha, void *o, int BH,
                               int N, int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream)
{
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    return dtype == LA_F32 ? by_dk<float>(q, k, v, alpha, o, BH, N, dk, dv, eps, stream)
                           : by_dk<__nv_bfloat16>(q, k, v, alpha, o, BH, N, dk, dv, eps, stream);
}

}  // namespace la
