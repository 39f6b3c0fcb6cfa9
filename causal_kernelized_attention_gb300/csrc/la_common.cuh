// Shared device helpers of the linear-attention library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "la.h"
#include "la_internal.h"

namespace la {

// Error bits of a device status word.  Each translation unit whose kernels run
// bounded waits owns one such word (a file-scope __device__ variable) and
// exports a host function that reads and clears it.
enum : unsigned { kStatusTimeout = 1u };

// phi(x) = elu(x) + 1 with alpha = 1, i.e. x + 1 for x > 0 and exp(x) otherwise
// ("Linear Transformer: elu+1", aicassindra.com).  The exp branch only sees
// x <= 0, so it never overflows.
__device__ __forceinline__ float phi_accurate(float x) { return x > 0.f ? x + 1.f : expf(x); }
__device__ __forceinline__ float phi_fast(float x) { return x > 0.f ? x + 1.f : __expf(x); }

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f32(float x) { return x; }
    static __device__ __forceinline__ float from_f32(float x) { return x; }
    static __device__ __forceinline__ float phi(float x) { return phi_accurate(x); }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
    static __device__ __forceinline__ float phi(float x) { return phi_fast(x); }
};

// Feature-map variants (struct Variant, la_internal.h).
template <typename T>
__device__ __forceinline__ float phi_variant(float x, const Variant &v)
{
    return v.map == LA_PHI_RELU ? fmaxf(x, 0.f) + v.shift : v.map == LA_PHI_IDENTITY ? x + v.shift : Elem<T>::phi(x);
}
// The output scale: 1 / max(den, eps), or 1 without the normaliser.
__device__ __forceinline__ float out_scale(float den, float eps, const Variant &v)
{
    return v.normalize ? 1.f / fmaxf(den, eps) : 1.f;
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace la
