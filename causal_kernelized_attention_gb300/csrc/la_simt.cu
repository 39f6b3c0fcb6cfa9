// CUDA-core (SIMT, fp32 arithmetic) kernels: the fp32 causal and non-causal
// forwards and the prefix-state reduction.  Tensor cores are not used here:
// tf32 would miss the fp32 path's 1e-5 relative tolerance.
//
// Causal: one CTA per (b,h, 32-column slice of dv) sweeps the chunks in order,
// the running state S (dk x 32) and z in shared memory ("Linear Attention",
// aiwiki.thehackersbrain.dev, chunked form: quadratic and masked inside a chunk,
// recurrent across chunks).
//
// The same kernel, instantiated with kDecay, computes the decayed state
// ("Linear Attention -- Math + Variants", RetNet and gated linear attention:
// S_t = g S_{t-1} + phi(k_t) v_t^T, z likewise, g a scalar per head).  In
// chunked form, with powers gp[d] = g^d of the per-head g:
//   intra-chunk score (a, b <= a)   * gp[a - b]
//   inter-chunk terms phi(q_a).S, phi(q_a).z   * gp[a + 1]
//   state after the chunk: gp[len] S + sum_j gp[len - 1 - j] phi(k_j) v_j^T, z likewise.
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kDVS = 32;  // dv columns per CTA (one per lane)

template <typename T, int DK, int C>
struct CausalSmem {
    float fk[C][DK + 1];   // phi(K_c), padded: lane j reads row j
    float vs[C][kDVS];     // V_c slice
    float S[DK][kDVS];     // running state slice, sum over earlier chunks
    float z[DK];           // running normaliser
    float qrow[kWarps][DK];
    float gp[C + 1];       // decay powers g^0 .. g^C (decayed form only)
};

// g^d, evaluated in double and rounded once to fp32 (g^0 = 1 for any g).  It is
// evaluated at most once per token or chunk offset, so the fp64 rate is immaterial.
__device__ __forceinline__ float decay_pow(float g, int d)
{
    return d == 0 ? 1.f : (float)pow((double)g, (double)d);
}

// Grid: (BH, dv / 32).  Block: 256 threads.  kDecay: g = gamma[bh % H].
template <typename T, int DK, int C, bool kDecay>
__global__ void __launch_bounds__(kThreads)
causal_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   T *__restrict__ o, int N, int DV, float eps, const float *__restrict__ gamma, int H,
                   const Variant var)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<CausalSmem<T, DK, C> *>(smem_raw);
    const int bh = blockIdx.x;
    const int c0 = blockIdx.y * kDVS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *qh = q + (size_t)bh * N * DK;
    const T *kh = k + (size_t)bh * N * DK;
    const T *vh = v + (size_t)bh * N * DV;
    T *oh = o + (size_t)bh * N * DV;

    for (int e = tid; e < DK * kDVS; e += kThreads) (&sm.S[0][0])[e] = 0.f;
    for (int e = tid; e < DK; e += kThreads) sm.z[e] = 0.f;
    if (kDecay) {
        const float g = gamma[bh % H];
        for (int d = tid; d <= C; d += kThreads) sm.gp[d] = decay_pow(g, d);
    }

    for (int i0 = 0; i0 < N; i0 += C) {
        const int len = min(C, N - i0);
        __syncthreads();  // previous chunk's state update is complete
        for (int e = tid; e < C * DK; e += kThreads) {
            const int j = e / DK, r = e % DK;
            sm.fk[j][r] = j < len ? phi_variant<T>(Elem<T>::to_f32(kh[(size_t)(i0 + j) * DK + r]), var) : 0.f;
        }
        for (int e = tid; e < C * kDVS; e += kThreads) {
            const int j = e / kDVS, c = e % kDVS;
            sm.vs[j][c] = (j < len && c0 + c < DV) ? Elem<T>::to_f32(vh[(size_t)(i0 + j) * DV + c0 + c]) : 0.f;
        }
        __syncthreads();

        // Outputs: one warp per query row, lanes over key positions then over columns.
        for (int a = warp; a < len; a += kWarps) {
            for (int r = lane; r < DK; r += 32)
                sm.qrow[warp][r] = phi_variant<T>(Elem<T>::to_f32(qh[(size_t)(i0 + a) * DK + r]), var);
            __syncwarp();
            // inter-chunk part: phi(q) . S (state of earlier chunks), phi(q) . z
            float num = 0.f, den = 0.f;
#pragma unroll 8
            for (int r = 0; r < DK; ++r) num += sm.qrow[warp][r] * sm.S[r][lane];
            for (int r = lane; r < DK; r += 32) den += sm.qrow[warp][r] * sm.z[r];
            if (kDecay) {
                num *= sm.gp[a + 1];
                den *= sm.gp[a + 1];
            }
            // intra-chunk part: scores s_ab = phi(q_a) . phi(k_b), b <= a (inclusive)
            float s[C / 32];
#pragma unroll
            for (int m = 0; m < C / 32; ++m) {
                const int b = lane + 32 * m;
                float acc = 0.f;
#pragma unroll 8
                for (int r = 0; r < DK; ++r) acc += sm.qrow[warp][r] * sm.fk[b][r];
                s[m] = (b <= a) ? (kDecay ? acc * sm.gp[a - b] : acc) : 0.f;
                den += s[m];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
#pragma unroll
            for (int m = 0; m < C / 32; ++m) {
                const int bmax = min(32, a + 1 - 32 * m);
                for (int bb = 0; bb < bmax; ++bb)
                    num += __shfl_sync(0xffffffffu, s[m], bb) * sm.vs[32 * m + bb][lane];
            }
            if (c0 + lane < DV)
                oh[(size_t)(i0 + a) * DV + c0 + lane] = Elem<T>::from_f32(var.normalize ? num / fmaxf(den, eps) : num);
            __syncwarp();
        }
        __syncthreads();

        // State update: S += phi(K_c)^T V_c, z += column sums of phi(K_c)
        // (decayed: the old state scaled by g^len, token j by g^(len-1-j)).
        for (int e = tid; e < DK * kDVS; e += kThreads) {
            const int r = e / kDVS, c = e % kDVS;
            float acc = kDecay ? sm.S[r][c] * sm.gp[len] : sm.S[r][c];
            for (int j = 0; j < len; ++j)
                acc += (kDecay ? sm.fk[j][r] * sm.gp[len - 1 - j] : sm.fk[j][r]) * sm.vs[j][c];
            sm.S[r][c] = acc;
        }
        for (int r = tid; r < DK; r += kThreads) {
            float acc = kDecay ? sm.z[r] * sm.gp[len] : sm.z[r];
            for (int j = 0; j < len; ++j) acc += kDecay ? sm.fk[j][r] * sm.gp[len - 1 - j] : sm.fk[j][r];
            sm.z[r] = acc;
        }
    }
}

// Partial prefix states: grid (BH, dv/32, splits).  Each CTA sums phi(k_t) v_t^T over
// its token range and adds the result into S (and z, from the first column slice)
// with atomics; S and z must be zero on entry.  kDecay: token t is weighted by
// g^(N-1-t), g = gamma[bh % H] (the decayed recurrence unrolled over the prefix).
constexpr int kStateTile = 64;

template <typename T, int DK, bool kDecay>
__global__ void __launch_bounds__(kThreads)
state_simt_kernel(const T *__restrict__ k, const T *__restrict__ v, float *__restrict__ S,
                  float *__restrict__ z, int N, int DV, int tokens_per_split,
                  const float *__restrict__ gamma, int H, const Variant var)
{
    __shared__ float fk[kStateTile][DK];
    __shared__ float vs[kStateTile][kDVS];
    __shared__ float wt[kStateTile];
    const int bh = blockIdx.x, c0 = blockIdx.y * kDVS;
    const int t0 = blockIdx.z * tokens_per_split;
    const int t1 = min(N, t0 + tokens_per_split);
    const int tid = threadIdx.x;
    const T *kh = k + (size_t)bh * N * DK;
    const T *vh = v + (size_t)bh * N * DV;
    constexpr int kPer = DK * kDVS / kThreads;  // state elements per thread
    float acc[kPer];
    float zacc = 0.f;
#pragma unroll
    for (int m = 0; m < kPer; ++m) acc[m] = 0.f;
    for (int b0 = t0; b0 < t1; b0 += kStateTile) {
        const int len = min(kStateTile, t1 - b0);
        __syncthreads();
        if (kDecay) {
            if (tid < kStateTile) wt[tid] = tid < len ? decay_pow(gamma[bh % H], N - 1 - (b0 + tid)) : 0.f;
            __syncthreads();
        }
        for (int e = tid; e < kStateTile * DK; e += kThreads) {
            const int j = e / DK, r = e % DK;
            float f = j < len ? phi_variant<T>(Elem<T>::to_f32(kh[(size_t)(b0 + j) * DK + r]), var) : 0.f;
            if (kDecay) f *= wt[j];
            fk[j][r] = f;
        }
        for (int e = tid; e < kStateTile * kDVS; e += kThreads) {
            const int j = e / kDVS, c = e % kDVS;
            vs[j][c] = (j < len && c0 + c < DV) ? Elem<T>::to_f32(vh[(size_t)(b0 + j) * DV + c0 + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kPer; ++m) {
            const int e = tid + m * kThreads, r = e / kDVS, c = e % kDVS;
            float a = acc[m];
            for (int j = 0; j < len; ++j) a += fk[j][r] * vs[j][c];
            acc[m] = a;
        }
        if (blockIdx.y == 0 && tid < DK)
            for (int j = 0; j < len; ++j) zacc += fk[j][tid];
    }
    float *Sh = S + (size_t)bh * DK * DV;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
        const int e = tid + m * kThreads, r = e / kDVS, c = e % kDVS;
        if (c0 + c < DV) atomicAdd(&Sh[(size_t)r * DV + c0 + c], acc[m]);
    }
    if (blockIdx.y == 0 && tid < DK) atomicAdd(&z[(size_t)bh * DK + tid], zacc);
}

// o = phi(Q) S / max(phi(Q) z, eps): grid (ceil(N/64), BH, dv/32); one warp per row.
template <typename T, int DK>
__global__ void __launch_bounds__(kThreads)
apply_simt_kernel(const T *__restrict__ q, const float *__restrict__ S, const float *__restrict__ z,
                  T *__restrict__ o, int N, int DV, float eps, const Variant var)
{
    __shared__ float Ss[DK][kDVS];
    __shared__ float zs[DK];
    __shared__ float qrow[kWarps][DK];
    const int bh = blockIdx.y, c0 = blockIdx.z * kDVS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *Sh = S + (size_t)bh * DK * DV;
    for (int e = tid; e < DK * kDVS; e += kThreads) {
        const int r = e / kDVS, c = e % kDVS;
        Ss[r][c] = c0 + c < DV ? Sh[(size_t)r * DV + c0 + c] : 0.f;
    }
    for (int r = tid; r < DK; r += kThreads) zs[r] = z[(size_t)bh * DK + r];
    __syncthreads();
    const T *qh = q + (size_t)bh * N * DK;
    T *oh = o + (size_t)bh * N * DV;
    const int row_end = min(N, (int)(blockIdx.x + 1) * 64);
    for (int i = blockIdx.x * 64 + warp; i < row_end; i += kWarps) {
        for (int r = lane; r < DK; r += 32) qrow[warp][r] = phi_variant<T>(Elem<T>::to_f32(qh[(size_t)i * DK + r]), var);
        __syncwarp();
        float num = 0.f, den = 0.f;
#pragma unroll 8
        for (int r = 0; r < DK; ++r) num += qrow[warp][r] * Ss[r][lane];
        for (int r = lane; r < DK; r += 32) den += qrow[warp][r] * zs[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        if (c0 + lane < DV) oh[(size_t)i * DV + c0 + lane] = Elem<T>::from_f32(var.normalize ? num / fmaxf(den, eps) : num);
        __syncwarp();
    }
}

template <typename T, int DK, int C>
la_status launch_causal(const Problem &p)
{
    const size_t smem = sizeof(CausalSmem<T, DK, C>);
    auto kern = p.gamma ? causal_simt_kernel<T, DK, C, true> : causal_simt_kernel<T, DK, C, false>;
    la_status st = ensure_smem((const void *)kern, (int)smem);
    if (st != LA_OK) return st;
    dim3 grid(p.BH, ceil_div(p.dv, kDVS));
    count_launches();
    kern<<<grid, kThreads, smem, p.stream>>>((const T *)p.q, (const T *)p.k, (const T *)p.v, (T *)p.o,
                                             p.N, p.dv, p.eps, p.gamma, p.H, p.var);
    return cuda_status(cudaGetLastError());
}

template <typename T, int DK>
la_status launch_state(const void *k, const void *v, float *S, float *z, int BH, int N, int dv,
                       cudaStream_t stream, const float *gamma = nullptr, int H = 1, Variant var = Variant())
{
    cudaError_t e = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)BH * DK * dv, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(z, 0, sizeof(float) * (size_t)BH * DK, stream);
    count_launches(2);
    if (e != cudaSuccess) return cuda_status(e);
    if (N == 0) return LA_OK;
    const int slices = ceil_div(dv, kDVS);
    // enough CTAs to cover the GPU a few times over, at least 256 tokens each
    int splits = ceil_div(4 * 152, BH * slices);
    splits = max(1, min(splits, ceil_div(N, 256)));
    const int per = ceil_div(ceil_div(N, splits), kStateTile) * kStateTile;
    splits = ceil_div(N, per);
    count_launches();
    if (gamma)
        state_simt_kernel<T, DK, true><<<dim3(BH, slices, splits), kThreads, 0, stream>>>(
            (const T *)k, (const T *)v, S, z, N, dv, per, gamma, H, var);
    else
        state_simt_kernel<T, DK, false><<<dim3(BH, slices, splits), kThreads, 0, stream>>>(
            (const T *)k, (const T *)v, S, z, N, dv, per, nullptr, 1, var);
    return cuda_status(cudaGetLastError());
}

template <typename T, int DK>
la_status launch_noncausal(const Problem &p)
{
    Scratch scratch;
    const size_t s_elems = (size_t)p.BH * DK * p.dv, z_elems = (size_t)p.BH * DK;
    la_status st = scratch.alloc(sizeof(float) * (s_elems + z_elems), p.stream);
    if (st != LA_OK) return st;
    float *S = (float *)scratch.ptr, *z = S + s_elems;
    st = launch_state<T, DK>(p.k, p.v, S, z, p.BH, p.N, p.dv, p.stream, nullptr, 1, p.var);
    if (st != LA_OK) return st;
    dim3 grid(ceil_div(p.N, 64), p.BH, ceil_div(p.dv, kDVS));
    count_launches();
    apply_simt_kernel<T, DK><<<grid, kThreads, 0, p.stream>>>((const T *)p.q, S, z, (T *)p.o, p.N, p.dv, p.eps,
                                                              p.var);
    return cuda_status(cudaGetLastError());
}

template <typename T>
la_status causal_by_dk(const Problem &p)
{
    const bool c64 = p.chunk == 64;
    switch (p.dk) {
    case 32: return c64 ? launch_causal<T, 32, 64>(p) : launch_causal<T, 32, 128>(p);
    case 64: return c64 ? launch_causal<T, 64, 64>(p) : launch_causal<T, 64, 128>(p);
    case 128: return c64 ? launch_causal<T, 128, 64>(p) : launch_causal<T, 128, 128>(p);
    }
    return LA_ERR_UNSUPPORTED;
}

template <typename T>
la_status state_by_dk(const void *k, const void *v, float *S, float *z, int BH, int N, int dk, int dv,
                      cudaStream_t s, const float *gamma, int H, const Variant &var)
{
    switch (dk) {
    case 32: return launch_state<T, 32>(k, v, S, z, BH, N, dv, s, gamma, H, var);
    case 64: return launch_state<T, 64>(k, v, S, z, BH, N, dv, s, gamma, H, var);
    case 128: return launch_state<T, 128>(k, v, S, z, BH, N, dv, s, gamma, H, var);
    }
    return LA_ERR_UNSUPPORTED;
}

template <typename T>
la_status noncausal_by_dk(const Problem &p)
{
    switch (p.dk) {
    case 32: return launch_noncausal<T, 32>(p);
    case 64: return launch_noncausal<T, 64>(p);
    case 128: return launch_noncausal<T, 128>(p);
    }
    return LA_ERR_UNSUPPORTED;
}

}  // namespace

la_status causal_simt(const Problem &p)
{
    if (!supported_dim(p.dk) || !supported_dim(p.dv) || (p.chunk != 64 && p.chunk != 128))
        return LA_ERR_UNSUPPORTED;
    return p.dtype == LA_F32 ? causal_by_dk<float>(p) : causal_by_dk<__nv_bfloat16>(p);
}

la_status noncausal_simt(const Problem &p)
{
    if (!supported_dim(p.dk) || !supported_dim(p.dv)) return LA_ERR_UNSUPPORTED;
    return p.dtype == LA_F32 ? noncausal_by_dk<float>(p) : noncausal_by_dk<__nv_bfloat16>(p);
}

la_status state_simt(const void *k, const void *v, float *S, float *z, int BH, int N, int dk, int dv,
                     la_dtype dtype, cudaStream_t stream, const float *gamma, int H, const Variant &var)
{
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    return dtype == LA_F32 ? state_by_dk<float>(k, v, S, z, BH, N, dk, dv, stream, gamma, H, var)
                           : state_by_dk<__nv_bfloat16>(k, v, S, z, BH, N, dk, dv, stream, gamma, H, var);
}

}  // namespace la

// ---------------------------------------------------------------------------
// Allocation-free non-causal forward (la_forward_noncausal_noalloc).
//
// Same kernels as the non-causal path above, but the S and z partial sums live
// in a fixed array compiled into the library instead of stream-ordered scratch.
// The array is shared by every call on a device and keeps the previous call's
// contents; launch_state clears the part a call uses before accumulating.
// Calls whose work overlaps on the GPU (other streams, other host threads) race
// on it.
// ---------------------------------------------------------------------------
#include <mutex>
#include <unordered_map>

namespace la {
namespace {

static __device__ __align__(256) float g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// Device address of g_noalloc_scratch on the current device.  In host code the
// symbol is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and cached.
la_status noalloc_scratch(float **out)
{
    static std::mutex mu;
    static std::unordered_map<int, float *> addr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find(dev);
    if (it == addr.end()) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        it = addr.emplace(dev, (float *)p).first;
    }
    *out = it->second;
    return LA_OK;
}

template <typename T, int DK>
la_status launch_noncausal_noalloc(const Problem &p, float *scratch)
{
    const size_t s_elems = (size_t)p.BH * DK * p.dv;
    float *S = scratch, *z = scratch + s_elems;  // s_elems is a multiple of 4: z stays 16-byte aligned
    la_status st = launch_state<T, DK>(p.k, p.v, S, z, p.BH, p.N, p.dv, p.stream, nullptr, 1, p.var);
    if (st != LA_OK) return st;
    dim3 grid(ceil_div(p.N, 64), p.BH, ceil_div(p.dv, kDVS));
    count_launches();
    apply_simt_kernel<T, DK><<<grid, kThreads, 0, p.stream>>>((const T *)p.q, S, z, (T *)p.o, p.N, p.dv, p.eps,
                                                              p.var);
    return cuda_status(cudaGetLastError());
}

template <typename T>
la_status noncausal_noalloc_by_dk(const Problem &p, float *scratch)
{
    switch (p.dk) {
    case 32: return launch_noncausal_noalloc<T, 32>(p, scratch);
    case 64: return launch_noncausal_noalloc<T, 64>(p, scratch);
    case 128: return launch_noncausal_noalloc<T, 128>(p, scratch);
    }
    return LA_ERR_UNSUPPORTED;
}

}  // namespace

la_status noncausal_simt_noalloc(const Problem &p)
{
    if (!supported_dim(p.dk) || !supported_dim(p.dv)) return LA_ERR_UNSUPPORTED;
    const size_t need = sizeof(float) * (size_t)p.BH * p.dk * ((size_t)p.dv + 1);
    if (need > LA_NOALLOC_SCRATCH_BYTES) return LA_ERR_UNSUPPORTED;
    float *scratch = nullptr;
    la_status st = noalloc_scratch(&scratch);
    if (st != LA_OK) return st;
    return p.dtype == LA_F32 ? noncausal_noalloc_by_dk<float>(p, scratch)
                             : noncausal_noalloc_by_dk<__nv_bfloat16>(p, scratch);
}

}  // namespace la
