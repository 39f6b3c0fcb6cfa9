// Recurrent decode step ("Linear Attention", aiwiki.thehackersbrain.dev, "It is a
// linear RNN": a fixed dk x dv state, O(d^2) per token; "26. Linear (Kernelized)
// Attention", Step-by-Step steps 3-4: update with the rank-1 term, then read):
//
//   S += phi(k) v^T,  z += phi(k),  o = phi(q)^T S / max(phi(q)^T z, eps)
//
// The decayed step ("Linear Attention -- Math + Variants", RetNet and gated
// linear attention: a scalar decay per head on the recurrent state) scales the
// old state and normaliser first: S = g S + phi(k) v^T, z = g z + phi(k).
//
// The step is bound by HBM traffic on S (fp32 read + write, 2*4*dk*dv bytes per
// head).  One CTA per head: each thread owns 16-byte column groups (float4) of a
// few rows of S, issues all of its loads before any arithmetic (so a CTA keeps
// its whole 64 KB state slice in flight), writes the updated rows back with
// streaming stores, and the per-row partial numerators are reduced across row
// groups in shared memory.  z and the denominator use one warp-level reduction.
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kDecodeThreads = 256;

template <typename T>
__device__ __forceinline__ void load4(const T *p, float out[4]);
template <>
__device__ __forceinline__ void load4<float>(const float *p, float out[4])
{
    const float4 x = *reinterpret_cast<const float4 *>(p);
    out[0] = x.x; out[1] = x.y; out[2] = x.z; out[3] = x.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float out[4])
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
    const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    out[0] = fa.x; out[1] = fa.y; out[2] = fb.x; out[3] = fb.y;
}

__device__ __forceinline__ float4 ld_stream(const float4 *p)
{
    float4 r;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ void st_stream(float4 *p, float4 v)
{
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w) : "memory");
}

// Grid: one CTA per head (blockIdx.x = b*H + h).  kDecay: gamma[(b*H + h) % H]
// scales the old S and z.
template <typename T, int DK, int DV, bool kDecay, bool kVar>
__global__ void __launch_bounds__(kDecodeThreads)
decode_kernel(float *__restrict__ S, float *__restrict__ z, const T *__restrict__ q,
              const T *__restrict__ k, const T *__restrict__ v, T *__restrict__ o, float eps,
              const float *__restrict__ gamma, int H, const Variant var)
{
    constexpr int kCols4 = DV / 4;                       // float4 groups per row
    constexpr int kRowGroups = kDecodeThreads / kCols4;  // threads stacked over rows
    constexpr int kRows = DK / kRowGroups;               // rows per thread
    static_assert(kRows >= 1 && DK % kRowGroups == 0, "shape");
    __shared__ float fq[DK], fk[DK];
    __shared__ float4 part[kRowGroups][kCols4];
    __shared__ float red[kDecodeThreads / 32];

    const size_t head = blockIdx.x;
    const int tid = threadIdx.x;
    const int cg = tid % kCols4, rg = tid / kCols4;
    float4 *Sh = reinterpret_cast<float4 *>(S + head * DK * DV);

    // Issue the state loads first: they are the whole cost of the step.
    float4 s[kRows];
#pragma unroll
    for (int m = 0; m < kRows; ++m) s[m] = ld_stream(Sh + (size_t)(rg + m * kRowGroups) * kCols4 + cg);
    const float g = kDecay ? gamma[head % H] : 1.f;

    for (int r = tid; r < DK; r += kDecodeThreads) {
        if (kVar) {
            fq[r] = phi_variant<T>(Elem<T>::to_f32(q[head * DK + r]), var);
            fk[r] = phi_variant<T>(Elem<T>::to_f32(k[head * DK + r]), var);
        } else {
            fq[r] = Elem<T>::phi(Elem<T>::to_f32(q[head * DK + r]));
            fk[r] = Elem<T>::phi(Elem<T>::to_f32(k[head * DK + r]));
        }
    }
    float vc[4];
    load4<T>(v + head * DV + 4 * cg, vc);
    __syncthreads();

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
        const int r = rg + m * kRowGroups;
        const float a = fk[r], b = fq[r];
        float4 x = s[m];
        if (kDecay) {
            x.x *= g; x.y *= g; x.z *= g; x.w *= g;
        }
        x.x += a * vc[0]; x.y += a * vc[1]; x.z += a * vc[2]; x.w += a * vc[3];
        st_stream(Sh + (size_t)r * kCols4 + cg, x);
        acc.x += b * x.x; acc.y += b * x.y; acc.z += b * x.z; acc.w += b * x.w;
    }
    part[rg][cg] = acc;

    // z update and denominator phi(q) . z_new.
    float d = 0.f;
    for (int r = tid; r < DK; r += kDecodeThreads) {
        const float zn = (kDecay ? g * z[head * DK + r] : z[head * DK + r]) + fk[r];
        z[head * DK + r] = zn;
        d += fq[r] * zn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if ((tid & 31) == 0) red[tid >> 5] = d;
    __syncthreads();
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeThreads / 32; ++w) den += red[w];
    const float inv = (kVar && !var.normalize) ? 1.f : 1.f / fmaxf(den, eps);

    // Column sums of the row-group partials: thread t < DV produces o[t].
    if (tid < DV) {
        const int c4 = tid >> 2, lane4 = tid & 3;
        float num = 0.f;
#pragma unroll 8
        for (int g = 0; g < kRowGroups; ++g) {
            const float4 p = part[g][c4];
            num += lane4 == 0 ? p.x : lane4 == 1 ? p.y : lane4 == 2 ? p.z : p.w;
        }
        o[head * DV + tid] = Elem<T>::from_f32(num * inv);
    }
}

struct DecodeArgs {
    float *S, *z;
    const void *q, *k, *v;
    void *o;
    int BH;
    float eps;
    const float *gamma;
    int H;
    cudaStream_t stream;
    Variant var;
};

template <typename T, int DK, int DV>
la_status launch(const DecodeArgs &a)
{
    count_launches();
    auto kern = a.gamma ? (a.var.is_default() ? decode_kernel<T, DK, DV, true, false> : decode_kernel<T, DK, DV, true, true>)
                        : (a.var.is_default() ? decode_kernel<T, DK, DV, false, false> : decode_kernel<T, DK, DV, false, true>);
    kern<<<a.BH, kDecodeThreads, 0, a.stream>>>(a.S, a.z, (const T *)a.q, (const T *)a.k, (const T *)a.v, (T *)a.o,
                                                 a.eps, a.gamma, a.gamma ? a.H : 1, a.var);
    return cuda_status(cudaGetLastError());
}

template <typename T, int DK>
la_status by_dv(const DecodeArgs &a, int dv)
{
    switch (dv) {
    case 32: return launch<T, DK, 32>(a);
    case 64: return launch<T, DK, 64>(a);
    case 128: return launch<T, DK, 128>(a);
    }
    return LA_ERR_UNSUPPORTED;
}

template <typename T>
la_status by_dk(const DecodeArgs &a, int dk, int dv)
{
    switch (dk) {
    case 32: return by_dv<T, 32>(a, dv);
    case 64: return by_dv<T, 64>(a, dv);
    case 128: return by_dv<T, 128>(a, dv);
    }
    return LA_ERR_UNSUPPORTED;
}

}  // namespace

la_status decode_step(float *S, float *z, const void *q, const void *k, const void *v, void *o, int BH,
                      int dk, int dv, float eps, la_dtype dtype, cudaStream_t stream,
                      const float *gamma, int H, const Variant &var)
{
    if (!supported_dim(dk) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
    const DecodeArgs a{S, z, q, k, v, o, BH, eps, gamma, H, stream, var};
    return dtype == LA_F32 ? by_dk<float>(a, dk, dv) : by_dk<__nv_bfloat16>(a, dk, dv);
}

}  // namespace la
