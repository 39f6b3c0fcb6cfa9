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
// Chunk-parallel, five launches over (b,h, chunk of C tokens):
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

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int DK, int DV>
struct Chunk {
    static constexpr int C = (DK > 64 || DV > 64) ? 32 : 64;  // tokens per chunk
    static constexpr int E = DK * (DV + 1);                    // floats per chunk state
};

// phi'(x) for elu + 1 from phi(x): 1 where x > 0 (phi > 1), exp(x) = phi(x) otherwise.
__device__ __forceinline__ float dphi_from_phi(float f) { return fminf(f, 1.f); }

// 1. A_c = phi(K_c)^T [V_c | 1].  Grid (nC, BH).
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_chunk_state(const T *__restrict__ k, const T *__restrict__ v, float *__restrict__ buf, int N)
{
    using CH = Chunk<DK, DV>;
    constexpr int C = CH::C;
    __shared__ float fk[C][DK];
    __shared__ float vs[C][DV + 1];
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int t0 = c * C, len = min(C, N - t0);
    const T *kh = k + ((size_t)bh * N + t0) * DK;
    const T *vh = v + ((size_t)bh * N + t0) * DV;
    for (int e = tid; e < C * DK; e += kThreads) {
        const int j = e / DK, r = e % DK;
        fk[j][r] = j < len ? Elem<T>::phi(Elem<T>::to_f32(kh[(size_t)j * DK + r])) : 0.f;
    }
    for (int e = tid; e < C * (DV + 1); e += kThreads) {
        const int j = e / (DV + 1), cc = e % (DV + 1);
        vs[j][cc] = j < len ? (cc < DV ? Elem<T>::to_f32(vh[(size_t)j * DV + cc]) : 1.f) : 0.f;
    }
    __syncthreads();
    float *out = buf + ((size_t)bh * gridDim.x + c) * CH::E;
    for (int e = tid; e < CH::E; e += kThreads) {
        const int r = e / (DV + 1), cc = e % (DV + 1);
        float acc = 0.f;
#pragma unroll 8
        for (int j = 0; j < C; ++j) acc += fk[j][r] * vs[j][cc];
        out[e] = acc;
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
    for (int i = 0; i < nC; i += 8) {
        float x[8];
        const int m = min(8, nC - i);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (u < m) {
                const int c = reverse ? nC - 1 - (i + u) : i + u;
                x[u] = p[(long long)c * E];
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (u < m) {
                const int c = reverse ? nC - 1 - (i + u) : i + u;
                p[(long long)c * E] = run;
                run += x[u];
            }
        }
    }
}

template <int DK, int DV>
struct DqSmem {
    static constexpr int C = Chunk<DK, DV>::C;
    float P[DK][DV + 1];    // prefix state before the chunk: S, z in column DV
    float fq[C][DK + 1];
    float fk[C][DK + 1];
    float vs[C][DV + 1];
    float dn[C][DV + 1];    // dn, dd in column DV
};

// 3. dq, dn, dd and the reverse chunk state.  Grid (nC, BH), one warp per query row.
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_dq(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, const T *__restrict__ dout,
       T *__restrict__ dq, float *__restrict__ buf, float *__restrict__ dnbuf, int N, float eps)
{
    using CH = Chunk<DK, DV>;
    constexpr int C = CH::C;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<DqSmem<DK, DV> *>(smem_raw);
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = c * C, len = min(C, N - t0);
    const size_t qk0 = ((size_t)bh * N + t0) * DK, v0 = ((size_t)bh * N + t0) * DV;
    float *slot = buf + ((size_t)bh * gridDim.x + c) * CH::E;
    for (int e = tid; e < CH::E; e += kThreads) sm.P[e / (DV + 1)][e % (DV + 1)] = slot[e];
    for (int e = tid; e < C * DK; e += kThreads) {
        const int j = e / DK, r = e % DK;
        sm.fq[j][r] = j < len ? Elem<T>::phi(Elem<T>::to_f32(q[qk0 + (size_t)j * DK + r])) : 0.f;
        sm.fk[j][r] = j < len ? Elem<T>::phi(Elem<T>::to_f32(k[qk0 + (size_t)j * DK + r])) : 0.f;
    }
    for (int e = tid; e < C * DV; e += kThreads) {
        const int j = e / DV, cc = e % DV;
        sm.vs[j][cc] = j < len ? Elem<T>::to_f32(v[v0 + (size_t)j * DV + cc]) : 0.f;
    }
    __syncthreads();

    constexpr int KB = C / 32;   // key blocks of 32 in the chunk
    for (int a = warp; a < len; a += kWarps) {
        // intra-chunk scores s_ab, b <= a (lane b of block m holds key 32m + lane)
        float s[KB];
        float den = 0.f;
#pragma unroll
        for (int m = 0; m < KB; ++m) {
            const int b = 32 * m + lane;
            float acc = 0.f;
#pragma unroll 8
            for (int r = 0; r < DK; ++r) acc += sm.fq[a][r] * sm.fk[b][r];
            s[m] = b <= a ? acc : 0.f;
            den += s[m];
        }
        for (int r = lane; r < DK; r += 32) den += sm.fq[a][r] * sm.P[r][DV];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        const bool clamped = !(den > eps);
        const float d = fmaxf(den, eps), inv = 1.f / d;
        // numerator columns, lanes over columns: n = phi(q_a) P + sum_b s_ab v_b
        float g = 0.f;
        for (int cc = lane; cc < DV; cc += 32) {
            float n = 0.f;
#pragma unroll 8
            for (int r = 0; r < DK; ++r) n += sm.fq[a][r] * sm.P[r][cc];
#pragma unroll
            for (int m = 0; m < KB; ++m) {
                const int bmax = min(32, a + 1 - 32 * m);
                for (int bb = 0; bb < bmax; ++bb) n += __shfl_sync(0xffffffffu, s[m], bb) * sm.vs[32 * m + bb][cc];
            }
            const float go = Elem<T>::to_f32(dout[v0 + (size_t)a * DV + cc]);
            g += go * (n * inv);
            sm.dn[a][cc] = go * inv;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) g += __shfl_xor_sync(0xffffffffu, g, off);
        const float dd = clamped ? 0.f : -g * inv;
        if (lane == 0) sm.dn[a][DV] = dd;
        __syncwarp();
        // t_b = v_b . dn_a + dd for the keys b <= a
        float tb[KB];
#pragma unroll
        for (int m = 0; m < KB; ++m) {
            const int b = 32 * m + lane;
            float acc = dd;
#pragma unroll 8
            for (int cc = 0; cc < DV; ++cc) acc += sm.vs[b][cc] * sm.dn[a][cc];
            tb[m] = b <= a ? acc : 0.f;
        }
        // dphi(q_a)[r] = P[r][:] . dn_a + dd z[r] + sum_b t_b phi(k_b)[r]
        for (int r = lane; r < DK; r += 32) {
            float acc = dd * sm.P[r][DV];
#pragma unroll 8
            for (int cc = 0; cc < DV; ++cc) acc += sm.P[r][cc] * sm.dn[a][cc];
#pragma unroll
            for (int m = 0; m < KB; ++m) {
                const int bmax = min(32, a + 1 - 32 * m);
                for (int bb = 0; bb < bmax; ++bb) acc += __shfl_sync(0xffffffffu, tb[m], bb) * sm.fk[32 * m + bb][r];
            }
            dq[qk0 + (size_t)a * DK + r] = Elem<T>::from_f32(acc * dphi_from_phi(sm.fq[a][r]));
        }
        float *dnrow = dnbuf + ((size_t)bh * N + t0 + a) * (DV + 1);
        for (int cc = lane; cc <= DV; cc += 32) dnrow[cc] = sm.dn[a][cc];
    }
    // rows past the end of the sequence contribute nothing to the reverse state
    for (int e = tid; e < (C - len) * (DV + 1); e += kThreads) sm.dn[len + e / (DV + 1)][e % (DV + 1)] = 0.f;
    __syncthreads();
    // B_c = phi(Q_c)^T [dN_c | dd_c] into this chunk's slot (the prefix was read above)
    for (int e = tid; e < CH::E; e += kThreads) {
        const int r = e / (DV + 1), cc = e % (DV + 1);
        float acc = 0.f;
#pragma unroll 8
        for (int a = 0; a < C; ++a) acc += sm.fq[a][r] * sm.dn[a][cc];
        slot[e] = acc;
    }
}

// 5. dk, dv.  Grid (nC, BH), one warp per key row.  Reuses the dq kernel's shared layout:
// P holds the suffix state [R | r] after the chunk.
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_dkdv(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, T *__restrict__ dk,
         T *__restrict__ dv, const float *__restrict__ buf, const float *__restrict__ dnbuf, int N)
{
    using CH = Chunk<DK, DV>;
    constexpr int C = CH::C;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<DqSmem<DK, DV> *>(smem_raw);
    const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = c * C, len = min(C, N - t0);
    const size_t qk0 = ((size_t)bh * N + t0) * DK, v0 = ((size_t)bh * N + t0) * DV;
    const float *slot = buf + ((size_t)bh * gridDim.x + c) * CH::E;
    for (int e = tid; e < CH::E; e += kThreads) sm.P[e / (DV + 1)][e % (DV + 1)] = slot[e];
    for (int e = tid; e < C * DK; e += kThreads) {
        const int j = e / DK, r = e % DK;
        sm.fq[j][r] = j < len ? Elem<T>::phi(Elem<T>::to_f32(q[qk0 + (size_t)j * DK + r])) : 0.f;
        sm.fk[j][r] = j < len ? Elem<T>::phi(Elem<T>::to_f32(k[qk0 + (size_t)j * DK + r])) : 0.f;
    }
    for (int e = tid; e < C * DV; e += kThreads) {
        const int j = e / DV, cc = e % DV;
        sm.vs[j][cc] = j < len ? Elem<T>::to_f32(v[v0 + (size_t)j * DV + cc]) : 0.f;
    }
    const float *dnc = dnbuf + ((size_t)bh * N + t0) * (DV + 1);
    for (int e = tid; e < C * (DV + 1); e += kThreads) {
        const int j = e / (DV + 1), cc = e % (DV + 1);
        sm.dn[j][cc] = j < len ? dnc[(size_t)j * (DV + 1) + cc] : 0.f;
    }
    __syncthreads();

    constexpr int KB = C / 32;
    for (int j = warp; j < len; j += kWarps) {
        // for the queries a >= j: u_a = dn_a . v_j + dd_a, w_a = phi(q_a) . phi(k_j)
        float u[KB], w[KB];
#pragma unroll
        for (int m = 0; m < KB; ++m) {
            const int a = 32 * m + lane;
            float au = sm.dn[a][DV], aw = 0.f;
#pragma unroll 8
            for (int cc = 0; cc < DV; ++cc) au += sm.dn[a][cc] * sm.vs[j][cc];
#pragma unroll 8
            for (int r = 0; r < DK; ++r) aw += sm.fq[a][r] * sm.fk[j][r];
            const bool in = a >= j && a < len;
            u[m] = in ? au : 0.f;
            w[m] = in ? aw : 0.f;
        }
        // dphi(k_j)[r] = R[r][:] . v_j + r[r] + sum_a u_a phi(q_a)[r]
        for (int r = lane; r < DK; r += 32) {
            float acc = sm.P[r][DV];
#pragma unroll 8
            for (int cc = 0; cc < DV; ++cc) acc += sm.P[r][cc] * sm.vs[j][cc];
#pragma unroll
            for (int m = 0; m < KB; ++m)
                for (int aa = 0; aa < 32; ++aa) acc += __shfl_sync(0xffffffffu, u[m], aa) * sm.fq[32 * m + aa][r];
            dk[qk0 + (size_t)j * DK + r] = Elem<T>::from_f32(acc * dphi_from_phi(sm.fk[j][r]));
        }
        // dv_j[cc] = R[:][cc] . phi(k_j) + sum_a w_a dn_a[cc]
        for (int cc = lane; cc < DV; cc += 32) {
            float acc = 0.f;
#pragma unroll 8
            for (int r = 0; r < DK; ++r) acc += sm.P[r][cc] * sm.fk[j][r];
#pragma unroll
            for (int m = 0; m < KB; ++m)
                for (int aa = 0; aa < 32; ++aa) acc += __shfl_sync(0xffffffffu, w[m], aa) * sm.dn[32 * m + aa][cc];
            dv[v0 + (size_t)j * DV + cc] = Elem<T>::from_f32(acc);
        }
    }
}

template <typename T, int DK, int DV>
la_status launch_backward(const BackwardProblem &p)
{
    using CH = Chunk<DK, DV>;
    const int nC = ceil_div(p.N, CH::C);
    const size_t state_floats = (size_t)p.BH * nC * CH::E;
    const size_t dn_floats = (size_t)p.BH * p.N * (DV + 1);
    Scratch scratch;
    la_status st = scratch.alloc(sizeof(float) * (state_floats + dn_floats), p.stream);
    if (st != LA_OK) return st;
    float *buf = (float *)scratch.ptr, *dnbuf = buf + state_floats;
    const size_t smem = sizeof(DqSmem<DK, DV>);
    st = ensure_smem((const void *)bwd_dq<T, DK, DV>, (int)smem);
    if (st == LA_OK) st = ensure_smem((const void *)bwd_dkdv<T, DK, DV>, (int)smem);
    if (st != LA_OK) return st;
    const dim3 grid(nC, p.BH);
    const long long total = (long long)p.BH * CH::E;
    const unsigned scan_blocks = (unsigned)((total + kThreads - 1) / kThreads);
    count_launches(5);
    bwd_chunk_state<T, DK, DV><<<grid, kThreads, 0, p.stream>>>((const T *)p.k, (const T *)p.v, buf, p.N);
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
    return p.dtype == LA_F32 ? backward_by_dk<float>(p) : backward_by_dk<__nv_bfloat16>(p);
}

}  // namespace la
