// Backward pass of the causal form (elu + 1, with the normaliser), CUDA cores, fp32.
//
// The pages give no gradient ("Linear Attention -- Math + Variants", Chunkwise
// parallelism: training runs the chunked form); this is the chain rule through the
// definition.  With n_i = phi(q_i)^T S_i, d_i = max(phi(q_i)^T z_i, eps), o_i = n_i / d_i
// and L = sum_i dO_i . o_i:
//
//   dn_i = dO_i / d_i,   dd_i = -(dO_i . o_i) / d_i   (0 where the clamp binds)
//   dphi(q_i) = S_i dn_i + dd_i z_i                                  (inclusive S_i, z_i)
//   dphi(k_j) = R_j v_j + r_j,   dv_j = R_j^T phi(k_j)
//   R_j = sum_{i>=j} phi(q_i) dn_i^T,   r_j = sum_{i>=j} dd_i phi(q_i)
//   dq = dphi(q) * phi'(q),  phi'(x) = 1 (x > 0), exp(x) (x <= 0) = min(1, phi(x)).
//
// Chunk-parallel, five launches over (b,h, chunk of C tokens); within a chunk every
// product is a block matrix product over the chunk's shared-memory tiles (a 16 x 16
// thread grid, each thread a register tile of the output):
//   1. chunk states    A_c = phi(K_c)^T [V_c | 1]                       -> buf[c]
//   2. forward scan    buf[c] = sum_{c' < c} A_c'   (exclusive prefix: S, z before c)
//   3. dq              per chunk: o, d, dn, dd, dq from the prefix and the intra-chunk
//                      scores; dn and dd to scratch; B_c = phi(Q_c)^T [dN_c | dd_c]
//                      over the chunk's own slot (no other CTA reads it)
//   4. reverse scan    buf[c] = sum_{c' > c} B_c'   (exclusive suffix: R, r after c)
//   5. dk, dv          per chunk from the suffix and the intra-chunk terms.
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;  // a 16 x 16 thread grid over every output tile

template <int DK, int DV>
struct Chunk {
    static constexpr int C = (DK > 64 || DV > 64) ? 32 : 64;  // tokens per chunk
    static constexpr int E = DK * (DV + 1);                    // floats per chunk state
};

// Shared-memory tiles of one chunk, fp32, rows padded by four floats: every row starts
// on a 16-byte boundary, and with row strides of 4 (mod 32) words the products' accesses
// -- 16 consecutive elements of a row, one address per half-warp, or one 16-byte vector
// from each of 8 consecutive rows per quarter-warp -- fall in distinct banks.
template <int DK, int DV>
struct Tiles {
    static constexpr int C = Chunk<DK, DV>::C;
    static constexpr int LQ = DK + 4, LV = DV + 4, LT = C + 4;
    static constexpr int kFq = 0;                 // phi(Q_c)        [C][LQ]
    static constexpr int kFk = kFq + C * LQ;      // phi(K_c)        [C][LQ]
    static constexpr int kV = kFk + C * LQ;       // V_c             [C][LV]
    static constexpr int kDn = kV + C * LV;       // [dN_c | dd_c]   [C][LV]
    static constexpr int kSt = kDn + C * LV;      // [S | z] or [R | r] of the chunk boundary  [DK][LV]
    static constexpr int kT = kSt + DK * LV;      // scores T, then U  [C][LT]
    static constexpr int kDen = kT + C * LT;      // denominators      [C]
    static constexpr int kFloats = kDen + C;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
    // the chunk-state kernel needs phi(K_c) and V_c only: [C][LQ] then [C][LV]
    static constexpr size_t kStateBytes = sizeof(float) * C * (LQ + LV);
};

// Operands of the products, element (r, k) of an R x K matrix in shared memory:
// KRow: k contiguous, at p[r * ld + k] (four consecutive k in one 16-byte load);
// KCol: r contiguous, at p[k * ld + r].
struct KRow {
    const float *p;
    int ld;
    __device__ __forceinline__ float4 load4(int r, int k) const
    {
        return *reinterpret_cast<const float4 *>(p + r * ld + k);
    }
};
struct KCol {
    const float *p;
    int ld;
    __device__ __forceinline__ float4 load4(int r, int k) const
    {
        return make_float4(p[k * ld + r], p[(k + 1) * ld + r], p[(k + 2) * ld + r], p[(k + 3) * ld + r]);
    }
};

// acc[i][j] += sum_k A(ty + 16 i, k) * B(tx + 16 j, k) for an M x N output on the 16 x 16
// thread grid (tx = thread % 16, ty = thread / 16); A is M x K and B is N x K (B(n, k) is
// element (k, n) of the right-hand factor), taken four k at a time.
template <int M, int N, int K, typename OA, typename OB>
__device__ __forceinline__ void gemm(float (&acc)[M / 16][N / 16], OA a, OB b)
{
    static_assert(K % 4 == 0, "K in steps of 4");
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 2
    for (int k = 0; k < K; k += 4) {
        float4 av[M / 16], bv[N / 16];
#pragma unroll
        for (int i = 0; i < M / 16; ++i) av[i] = a.load4(ty + 16 * i, k);
#pragma unroll
        for (int j = 0; j < N / 16; ++j) bv[j] = b.load4(tx + 16 * j, k);
#pragma unroll
        for (int i = 0; i < M / 16; ++i)
#pragma unroll
            for (int j = 0; j < N / 16; ++j) {
                acc[i][j] = fmaf(av[i].x, bv[j].x, acc[i][j]);
                acc[i][j] = fmaf(av[i].y, bv[j].y, acc[i][j]);
                acc[i][j] = fmaf(av[i].z, bv[j].z, acc[i][j]);
                acc[i][j] = fmaf(av[i].w, bv[j].w, acc[i][j]);
            }
    }
}

template <int M, int N>
__device__ __forceinline__ void zero(float (&acc)[M][N])
{
#pragma unroll
    for (int i = 0; i < M; ++i)
#pragma unroll
        for (int j = 0; j < N; ++j) acc[i][j] = 0.f;
}

// phi'(x) for elu + 1 from phi(x): 1 where x > 0 (phi > 1), exp(x) = phi(x) otherwise.
__device__ __forceinline__ float dphi_from_phi(float f) { return fminf(f, 1.f); }

// Rows [0, len) of a contiguous [rows x W] block of T elements into shared-memory rows
// of stride LD as fp32, through f (rows past len are zero).  Every 16-byte load of a
// thread is issued before any is used, so a tile costs one memory latency, not one
// per element.
template <typename T, int C, int W, typename F>
__device__ __forceinline__ void load_tile(float *dst, int LD, const T *src, int len, F f)
{
    constexpr int VE = 16 / (int)sizeof(T);  // elements per 16-byte vector
    constexpr int VR = W / VE;                // vectors per row
    constexpr int NV = C * VR;
    constexpr int IT = (NV + kThreads - 1) / kThreads;
    uint4 buf[IT];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int vi = threadIdx.x + it * kThreads;
        buf[it] = (vi < NV && vi / VR < len) ? __ldg(reinterpret_cast<const uint4 *>(src) + vi)
                                              : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int vi = threadIdx.x + it * kThreads;
        if (vi >= NV) break;
        const int row = vi / VR, col = (vi % VR) * VE;
        const T *e = reinterpret_cast<const T *>(&buf[it]);
#pragma unroll
        for (int u = 0; u < VE; ++u) dst[row * LD + col + u] = row < len ? f(Elem<T>::to_f32(e[u])) : 0.f;
    }
}

// Rows [0, rows) of W floats each, contiguous in global memory (any alignment), into
// shared-memory rows of stride LD; rows at or past `valid` read as zero.  Loads go in
// batches of 8 per thread, all issued before their stores.
template <int W>
__device__ __forceinline__ void load_rows(float *dst, int LD, const float *src, int rows, int valid)
{
    const int n = rows * W;
    for (int base = 0; base < n; base += 8 * kThreads) {
        float buf[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = base + (int)threadIdx.x + u * kThreads;
            buf[u] = (e < n && e / W < valid) ? __ldg(src + e) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = base + (int)threadIdx.x + u * kThreads;
            if (e < n) dst[(e / W) * LD + e % W] = buf[u];
        }
    }
}

// phi(Q_c), phi(K_c), V_c into their tiles (rows past the sequence zero).
template <typename T, int DK, int DV>
__device__ __forceinline__ void load_qkv(float *sm, const T *q, const T *k, const T *v, size_t qk0, size_t v0,
                                         int len)
{
    using L = Tiles<DK, DV>;
    auto phi = [](float x) { return Elem<T>::phi(x); };
    auto id = [](float x) { return x; };
    load_tile<T, L::C, DK>(sm + L::kFq, L::LQ, q + qk0, len, phi);
    load_tile<T, L::C, DK>(sm + L::kFk, L::LQ, k + qk0, len, phi);
    load_tile<T, L::C, DV>(sm + L::kV, L::LV, v + v0, len, id);
}

// T = phi(Q_c) phi(K_c)^T with the causal mask (key <= query < len) into the T tile.
template <int DK, int DV>
__device__ __forceinline__ void scores(float *sm, int len)
{
    using L = Tiles<DK, DV>;
    constexpr int C = L::C;
    const float *fq = sm + L::kFq, *fk = sm + L::kFk;
    float *ts = sm + L::kT;
    float acc[C / 16][C / 16];
    zero(acc);
    gemm<C, C, DK>(acc, KRow{fq, L::LQ}, KRow{fk, L::LQ});
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
    for (int i = 0; i < C / 16; ++i)
#pragma unroll
        for (int j = 0; j < C / 16; ++j) {
            const int m = ty + 16 * i, n = tx + 16 * j;
            ts[m * L::LT + n] = (n <= m && m < len) ? acc[i][j] : 0.f;
        }
}

// U = (dN_c V_c^T + dd_c 1^T) with the causal mask into the T tile.
template <int DK, int DV>
__device__ __forceinline__ void weights_u(float *sm, int len)
{
    using L = Tiles<DK, DV>;
    constexpr int C = L::C;
    const float *dn = sm + L::kDn, *vs = sm + L::kV;
    float *ts = sm + L::kT;
    float acc[C / 16][C / 16];
    zero(acc);
    gemm<C, C, DV>(acc, KRow{dn, L::LV}, KRow{vs, L::LV});
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
    for (int i = 0; i < C / 16; ++i) {
        const int m = ty + 16 * i;
        const float dd = dn[m * L::LV + DV];
#pragma unroll
        for (int j = 0; j < C / 16; ++j) {
            const int n = tx + 16 * j;
            ts[m * L::LT + n] = (n <= m && m < len) ? acc[i][j] + dd : 0.f;
        }
    }
}

// 1. A_c = phi(K_c)^T [V_c | 1] -> buf[c].  Grid (nC, BH).
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_chunk_state(const T *__restrict__ k, const T *__restrict__ v, float *__restrict__ buf, int N)
{
    using L = Tiles<DK, DV>;
    constexpr int C = L::C;
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int t0 = c * C, len = min(C, N - t0);
    const size_t qk0 = ((size_t)bh * N + t0) * DK, v0 = ((size_t)bh * N + t0) * DV;
    float *fk = sm, *vs = sm + C * L::LQ;  // the kStateBytes layout
    load_tile<T, C, DK>(fk, L::LQ, k + qk0, len, [](float x) { return Elem<T>::phi(x); });
    load_tile<T, C, DV>(vs, L::LV, v + v0, len, [](float x) { return x; });
    __syncthreads();
    float *out = buf + ((size_t)bh * gridDim.x + c) * Chunk<DK, DV>::E;
    float acc[DK / 16][DV / 16];
    zero(acc);
    gemm<DK, DV, C>(acc, KCol{fk, L::LQ}, KCol{vs, L::LV});
    const int tx = tid & 15, ty = tid >> 4;
#pragma unroll
    for (int i = 0; i < DK / 16; ++i)
#pragma unroll
        for (int j = 0; j < DV / 16; ++j) out[(ty + 16 * i) * (DV + 1) + tx + 16 * j] = acc[i][j];
    if (tid < DK) {  // z column: the column sums of phi(K_c)
        float s = 0.f;
        for (int kk = 0; kk < C; ++kk) s += fk[kk * L::LQ + tid];
        out[tid * (DV + 1) + DV] = s;
    }
}

// 2./4. Exclusive scan over the chunks of each head, in place: forward (prefix) or
// reverse (suffix).  Thread = (bh, element); consecutive threads, consecutive elements.
__global__ void __launch_bounds__(kThreads)
bwd_scan(float *__restrict__ buf, int nC, int E, long long total, int reverse)
{
    const long long g = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (g >= total) return;
    const long long bh = g / E, e = g % E;
    float *p = buf + bh * (long long)nC * E + e;
    float run = 0.f;
    // 32 chunks per round trip: every load of a round is issued before the first store
    for (int i = 0; i < nC; i += 32) {
        float x[32];
        const int m = min(32, nC - i);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            if (u < m) {
                const int c = reverse ? nC - 1 - (i + u) : i + u;
                x[u] = p[(long long)c * E];
            }
        }
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            if (u < m) {
                const int c = reverse ? nC - 1 - (i + u) : i + u;
                p[(long long)c * E] = run;
                run += x[u];
            }
        }
    }
}

// 3. Per chunk: o and the clamped denominator d, dN = dO / d and dd = -(dO . o) / d
// (0 where the clamp binds) to dnbuf, dq, and the reverse chunk state
// B_c = phi(Q_c)^T [dN_c | dd_c] over the chunk's own slot.  Grid (nC, BH).
//   T   = tril(phi(Q) phi(K)^T)          den = rowsum T + phi(Q) z
//   num = T V + phi(Q) S                 U   = tril(dN V^T + dd 1^T)
//   dphi(Q) = U phi(K) + dN S^T + dd z^T
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_dq(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, const T *__restrict__ dout,
       T *__restrict__ dq, float *__restrict__ buf, float *__restrict__ dnbuf, int N, float eps)
{
    using L = Tiles<DK, DV>;
    constexpr int C = L::C;
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int t0 = c * C, len = min(C, N - t0);
    const size_t qk0 = ((size_t)bh * N + t0) * DK, v0 = ((size_t)bh * N + t0) * DV;
    const float *fq = sm + L::kFq, *fk = sm + L::kFk, *vs = sm + L::kV, *st = sm + L::kSt, *ts = sm + L::kT;
    float *dn = sm + L::kDn, *den = sm + L::kDen;
    float *slot = buf + ((size_t)bh * gridDim.x + c) * Chunk<DK, DV>::E;
    load_rows<DV + 1>(sm + L::kSt, L::LV, slot, DK, DK);  // [S | z] before the chunk
    load_qkv<T, DK, DV>(sm, q, k, v, qk0, v0, len);
    // this thread's dO elements, in flight while the scores are formed
    float go[C / 16][DV / 16];
#pragma unroll
    for (int i = 0; i < C / 16; ++i)
#pragma unroll
        for (int j = 0; j < DV / 16; ++j) {
            const int m = ty + 16 * i;
            go[i][j] = m < len ? Elem<T>::to_f32(dout[v0 + (size_t)m * DV + tx + 16 * j]) : 0.f;
        }
    __syncthreads();
    scores<DK, DV>(sm, len);
    __syncthreads();
    if (tid < C) {
        float s = 0.f;
        for (int n = 0; n < C; ++n) s += ts[tid * L::LT + n];
        for (int r = 0; r < DK; ++r) s += fq[tid * L::LQ + r] * st[r * L::LV + DV];
        den[tid] = s;
    }
    __syncthreads();
    {
        float acc[C / 16][DV / 16];
        zero(acc);
        gemm<C, DV, C>(acc, KRow{ts, L::LT}, KCol{vs, L::LV});
        gemm<C, DV, DK>(acc, KRow{fq, L::LQ}, KCol{st, L::LV});
#pragma unroll
        for (int i = 0; i < C / 16; ++i) {
            const int m = ty + 16 * i;
            const float inv = 1.f / fmaxf(den[m], eps);
            float g = 0.f;
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) g += go[i][j] * (acc[i][j] * inv);
            // g = dO_m . o_m over the 16 threads of this row (lanes of one half-warp)
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) g += __shfl_xor_sync(0xffffffffu, g, off);
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) dn[m * L::LV + tx + 16 * j] = go[i][j] * inv;
            if (tx == 0) dn[m * L::LV + DV] = den[m] > eps ? -g * inv : 0.f;
        }
    }
    __syncthreads();
    {
        float *dst = dnbuf + ((size_t)bh * N + t0) * (DV + 1);
        for (int e = tid; e < len * (DV + 1); e += kThreads) dst[e] = dn[(e / (DV + 1)) * L::LV + e % (DV + 1)];
    }
    weights_u<DK, DV>(sm, len);
    __syncthreads();
    {
        float acc[C / 16][DK / 16];
        zero(acc);
        gemm<C, DK, C>(acc, KRow{ts, L::LT}, KCol{fk, L::LQ});
        gemm<C, DK, DV>(acc, KRow{dn, L::LV}, KRow{st, L::LV});
#pragma unroll
        for (int i = 0; i < C / 16; ++i) {
            const int m = ty + 16 * i;
            if (m >= len) continue;
            const float dd = dn[m * L::LV + DV];
#pragma unroll
            for (int j = 0; j < DK / 16; ++j) {
                const int n = tx + 16 * j;
                const float g = acc[i][j] + dd * st[n * L::LV + DV];
                dq[qk0 + (size_t)m * DK + n] = Elem<T>::from_f32(g * dphi_from_phi(fq[m * L::LQ + n]));
            }
        }
    }
    {
        // B_c (the slot's prefix was read into shared memory at the start)
        float acc[DK / 16][DV / 16];
        zero(acc);
        gemm<DK, DV, C>(acc, KCol{fq, L::LQ}, KCol{dn, L::LV});
#pragma unroll
        for (int i = 0; i < DK / 16; ++i)
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) slot[(ty + 16 * i) * (DV + 1) + tx + 16 * j] = acc[i][j];
        if (tid < DK) {
            float s = 0.f;
            for (int kk = 0; kk < C; ++kk) s += fq[kk * L::LQ + tid] * dn[kk * L::LV + DV];
            slot[tid * (DV + 1) + DV] = s;
        }
    }
}

// 5. dk, dv per chunk from the suffix [R | r] after it.  Grid (nC, BH).
//   dV      = T^T dN + phi(K) R
//   dphi(K) = U^T phi(Q) + V R^T + 1 r^T
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_dkdv(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, T *__restrict__ dk,
         T *__restrict__ dv, const float *__restrict__ buf, const float *__restrict__ dnbuf, int N)
{
    using L = Tiles<DK, DV>;
    constexpr int C = L::C;
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int t0 = c * C, len = min(C, N - t0);
    const size_t qk0 = ((size_t)bh * N + t0) * DK, v0 = ((size_t)bh * N + t0) * DV;
    const float *fq = sm + L::kFq, *fk = sm + L::kFk, *vs = sm + L::kV, *dn = sm + L::kDn, *st = sm + L::kSt,
                *ts = sm + L::kT;
    const float *slot = buf + ((size_t)bh * gridDim.x + c) * Chunk<DK, DV>::E;
    load_rows<DV + 1>(sm + L::kSt, L::LV, slot, DK, DK);  // [R | r] after the chunk
    load_qkv<T, DK, DV>(sm, q, k, v, qk0, v0, len);
    load_rows<DV + 1>(sm + L::kDn, L::LV, dnbuf + ((size_t)bh * N + t0) * (DV + 1), C, len);
    __syncthreads();
    scores<DK, DV>(sm, len);
    __syncthreads();
    {
        float acc[C / 16][DV / 16];
        zero(acc);
        gemm<C, DV, C>(acc, KCol{ts, L::LT}, KCol{dn, L::LV});
        gemm<C, DV, DK>(acc, KRow{fk, L::LQ}, KCol{st, L::LV});
#pragma unroll
        for (int i = 0; i < C / 16; ++i) {
            const int m = ty + 16 * i;
            if (m >= len) continue;
#pragma unroll
            for (int j = 0; j < DV / 16; ++j) dv[v0 + (size_t)m * DV + tx + 16 * j] = Elem<T>::from_f32(acc[i][j]);
        }
    }
    __syncthreads();  // the T tile is read; U replaces it
    weights_u<DK, DV>(sm, len);
    __syncthreads();
    {
        float acc[C / 16][DK / 16];
        zero(acc);
        gemm<C, DK, C>(acc, KCol{ts, L::LT}, KCol{fq, L::LQ});
        gemm<C, DK, DV>(acc, KRow{vs, L::LV}, KRow{st, L::LV});
#pragma unroll
        for (int i = 0; i < C / 16; ++i) {
            const int m = ty + 16 * i;
            if (m >= len) continue;
#pragma unroll
            for (int j = 0; j < DK / 16; ++j) {
                const int n = tx + 16 * j;
                const float g = acc[i][j] + st[n * L::LV + DV];
                dk[qk0 + (size_t)m * DK + n] = Elem<T>::from_f32(g * dphi_from_phi(fk[m * L::LQ + n]));
            }
        }
    }
}

template <typename T, int DK, int DV>
la_status launch_backward(const BackwardProblem &p)
{
    using CH = Chunk<DK, DV>;
    using L = Tiles<DK, DV>;
    const int nC = ceil_div(p.N, CH::C);
    const size_t state_floats = (size_t)p.BH * nC * CH::E;
    const size_t dn_floats = (size_t)p.BH * p.N * (DV + 1);
    Scratch scratch;
    la_status st = scratch.alloc(sizeof(float) * (state_floats + dn_floats), p.stream);
    if (st != LA_OK) return st;
    float *buf = (float *)scratch.ptr, *dnbuf = buf + state_floats;
    const int smem = (int)L::kBytes;
    st = ensure_smem((const void *)bwd_chunk_state<T, DK, DV>, (int)L::kStateBytes);
    if (st == LA_OK) st = ensure_smem((const void *)bwd_dq<T, DK, DV>, smem);
    if (st == LA_OK) st = ensure_smem((const void *)bwd_dkdv<T, DK, DV>, smem);
    if (st != LA_OK) return st;
    const dim3 grid(nC, p.BH);
    const long long total = (long long)p.BH * CH::E;
    const unsigned scan_blocks = (unsigned)((total + kThreads - 1) / kThreads);
    count_launches(5);
    bwd_chunk_state<T, DK, DV><<<grid, kThreads, L::kStateBytes, p.stream>>>((const T *)p.k, (const T *)p.v, buf,
                                                                             p.N);
    bwd_scan<<<scan_blocks, kThreads, 0, p.stream>>>(buf, nC, CH::E, total, 0);
    bwd_dq<T, DK, DV><<<grid, kThreads, smem, p.stream>>>((const T *)p.q, (const T *)p.k, (const T *)p.v,
                                                          (const T *)p.dout, (T *)p.dq, buf, dnbuf, p.N, p.eps);
    bwd_scan<<<scan_blocks, kThreads, 0, p.stream>>>(buf, nC, CH::E, total, 1);
    bwd_dkdv<T, DK, DV><<<grid, kThreads, smem, p.stream>>>((const T *)p.q, (const T *)p.k, (const T *)p.v,
                                                            (T *)p.dk, (T *)p.dv, buf, dnbuf, p.N);
    return cuda_status(cudaGetLastError());
}

template <typename T, int DK>
la_status backward_by_dv(const BackwardProblem &p)
{
    switch (p.dvd) {
    case 32: return launch_backward<T, DK, 32>(p);
    case 64: return launch_backward<T, DK, 64>(p);
    case 128: return launch_backward<T, DK, 128>(p);
    }
    return LA_ERR_UNSUPPORTED;
}

template <typename T>
la_status backward_by_dk(const BackwardProblem &p)
{
    switch (p.dkd) {
    case 32: return backward_by_dv<T, 32>(p);
    case 64: return backward_by_dv<T, 64>(p);
    case 128: return backward_by_dv<T, 128>(p);
    }
    return LA_ERR_UNSUPPORTED;
}

}  // namespace

la_status causal_backward(const BackwardProblem &p)
{
    if (!supported_dim(p.dkd) || !supported_dim(p.dvd)) return LA_ERR_UNSUPPORTED;
    if (backward_tc_eligible(p)) return causal_backward_tc(p);
    return p.dtype == LA_F32 ? backward_by_dk<float>(p) : backward_by_dk<__nv_bfloat16>(p);
}

}  // namespace la
