// Shared pieces of the tensor-core (tcgen05 + TMA) kernels: bounded waits,
// the phi feature map on swizzled bf16 tiles, shared-memory descriptors, the
// helpers that write the bf16 state copy and the z split, the thread-major
// state layout, and the host-side TMA tensor maps.
#pragma once

#include <cuda_bf16.h>

#include <mutex>
#include <unordered_map>

#include "la_common.cuh"
#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {
namespace tc {

using namespace sm100;

constexpr int kC = 128;                            // chunk (tokens per tile)
constexpr uint32_t kBox = kC * 128;                // one [128 rows x 64 bf16] swizzled box: 16 KB
constexpr uint32_t kSleepHintNs = 200000;          // per try_wait; the total wait stays bounded below
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any healthy wait

__device__ __forceinline__ bool aborted(const volatile int *a) { return *a != 0; }

// Bounded wait on an mbarrier phase; sets the CTA abort flag and the calling
// translation unit's device status word on expiry.
__device__ __forceinline__ bool wait_bar(unsigned *status, int *abort_flag, uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (aborted(abort_flag)) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *(volatile int *)abort_flag = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Same, with one result for the whole warp (for roles that issue warp-collective
// tcgen05.ld / tcgen05.st after the wait).
__device__ __forceinline__ bool wait_bar_warp(unsigned *status, int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, wait_bar(status, abort_flag, bar, parity));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// phi on a pair of bf16 values: exp(min(x, 0)) + max(x, 0), which is x + 1 for
// x > 0 and exp(x) otherwise, all in packed bf16x2: y = min(x, 0) * log2(e) with
// one rounding (log2(e) split into a bf16 head and tail, fused multiply-add),
// then the packed bf16 exp2 of the special-function unit (two values per
// operation), then the exact add of max(x, 0).  The result is a bf16 tensor-core
// operand either way; rounding y to bf16 perturbs exp(x) by at most
// 2^(|y| 2^-9) - 1 relative (about |x| 2^-9: 0.3% at x = -4, 9% at x = -30).
// On outputs that is invisible next to the bf16 rounding of phi and of the
// scores at any input scale (a uniform error in phi(q) cancels in the ratio);
// only where the clamp of the denominator binds does phi(q)'s error reach the
// output unscaled, and there the output is itself ~phi(q).S / eps, tiny.  An
// fp32 exponential (one more special-function operation per value) measured
// 1.25-1.5x slower causal forwards for no change in any output tolerance.
__device__ __forceinline__ uint32_t ex2_bf16x2(uint32_t y)
{
    uint32_t r;
    asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(r) : "r"(y));
    return r;
}
__device__ __forceinline__ uint32_t phi2(uint32_t w)
{
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&w);
    const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
    const __nv_bfloat162 log2e_hi = __float2bfloat162_rn(1.4453125f);          // bf16(log2 e)
    const __nv_bfloat162 log2e_lo = __float2bfloat162_rn(-0.0026174591f);      // log2 e - head
    const __nv_bfloat162 neg = __hmin2(x, zero);
    const __nv_bfloat162 y = __hfma2(neg, log2e_hi, __hmul2(neg, log2e_lo));
    const uint32_t yb = *reinterpret_cast<const uint32_t *>(&y);
    const uint32_t eb = ex2_bf16x2(yb);
    const __nv_bfloat162 r = __hadd2(*reinterpret_cast<const __nv_bfloat162 *>(&eb), __hmax2(x, zero));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Feature-map variants on a pair of bf16 values (map LA_PHI_RELU: max(x, 0) + c,
// LA_PHI_IDENTITY: x + c; LA_PHI_ELU1: phi2), in packed bf16: the max is exact and
// the add rounds once; c2 is the shift rounded to bf16 (2^-9 relative, the size of
// the operand's own rounding).
__device__ __forceinline__ uint32_t phi2_variant(uint32_t w, int map, uint32_t c2)
{
    if (map == LA_PHI_ELU1) return phi2(w);
    __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&w);
    if (map == LA_PHI_RELU) x = __hmax2(x, __float2bfloat162_rn(0.f));
    const __nv_bfloat162 r = __hadd2(x, *reinterpret_cast<const __nv_bfloat162 *>(&c2));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Decayed state: gamma^e for an integer e >= 0 from lg = log2(gamma) (gamma^0 = 1
// for any gamma, including 0, whose lg is -inf).
__device__ __forceinline__ float pow_decay(float lg, int e)
{
    return e == 0 ? 1.f : exp2f((float)e * lg);
}
// w times a pair of bf16 values: one packed bf16 multiply by w rounded to bf16
// (the weight's own rounding, 2^-9 relative, is the size of the operand's).
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, uint32_t w2)
{
    const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&v),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&w2));
    return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t bf16x2_splat(float w) { return pack_bf16(w, w); }
// Row `row` of a 128-row, 128-byte-swizzled bf16 tile of D columns (D / 64 boxes)
// multiplied by w in place (the swizzle permutes 16-byte chunks within the row, so
// any chunk order will do: rotated by the row, 8 consecutive rows hit 8 bank groups).
template <int D>
__device__ __forceinline__ void scale_row(uint8_t *tile, int row, float wf)
{
    const uint32_t w = bf16x2_splat(wf);
#pragma unroll
    for (int b = 0; b < D / 64; ++b) {
        uint4 *rp = reinterpret_cast<uint4 *>(tile + b * kBox + row * 128);
        uint4 x[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = rp[(c + row) & 7];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            rp[(c + row) & 7] = make_uint4(scale_bf16x2(x[c].x, w), scale_bf16x2(x[c].y, w),
                                           scale_bf16x2(x[c].z, w), scale_bf16x2(x[c].w, w));
    }
}

// phi in place on one shared-memory tile, by NT threads.  A unit is half of one
// 128-byte row of a 64-column box (4 chunks of 16 bytes); thread t takes units
// t, t + NT, ...  Units of rows >= `valid` (past the end of the sequence) are
// zeroed.  All loads of a thread are issued before its arithmetic.  The chunk
// order is rotated by the row so that the 8 threads of a quarter-warp (8
// consecutive rows) touch 8 different bank groups.
// kScale (decayed state): row r is also multiplied by gamma^(ebase - r), lg = log2(gamma).
// kVar: the feature map `map` with shift c (phi2_variant) instead of elu + 1.
template <int D, int NT, bool kScale = false, bool kVar = false>
__device__ __forceinline__ void phi_tile(uint8_t *tile, int t, int valid, float lg = 0.f, int ebase = 0,
                                         int map = LA_PHI_ELU1, float c = 0.f)
{
    constexpr int kUnits = 128 * (D / 32);
    constexpr int NU = (kUnits + NT - 1) / NT;
    const uint32_t c2 = kVar ? pack_bf16(c, c) : 0u;
    uint4 buf[NU][4];
#pragma unroll
    for (int m = 0; m < NU; ++m) {
        const int u = t + NT * m, row = u & 127, hb = u >> 7;
        if (u < kUnits) {
            const uint8_t *rp = tile + (hb >> 1) * kBox + row * 128;
            const int rot = row + (hb & 1) * 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) buf[m][k] = *reinterpret_cast<const uint4 *>(rp + ((rot + k) & 7) * 16);
        }
    }
#pragma unroll
    for (int m = 0; m < NU; ++m) {
        const int u = t + NT * m, row = u & 127;
        const uint32_t w = kScale ? bf16x2_splat(pow_decay(lg, ebase - row)) : 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 &x = buf[m][k];
            if (kVar)
                x = row < valid ? make_uint4(phi2_variant(x.x, map, c2), phi2_variant(x.y, map, c2),
                                             phi2_variant(x.z, map, c2), phi2_variant(x.w, map, c2))
                                : make_uint4(0u, 0u, 0u, 0u);
            else
                x = row < valid ? make_uint4(phi2(x.x), phi2(x.y), phi2(x.z), phi2(x.w)) : make_uint4(0u, 0u, 0u, 0u);
            if (kScale)
                x = make_uint4(scale_bf16x2(x.x, w), scale_bf16x2(x.y, w), scale_bf16x2(x.z, w), scale_bf16x2(x.w, w));
        }
    }
#pragma unroll
    for (int m = 0; m < NU; ++m) {
        const int u = t + NT * m, row = u & 127, hb = u >> 7;
        if (u < kUnits) {
            uint8_t *rp = tile + (hb >> 1) * kBox + row * 128;
            const int rot = row + (hb & 1) * 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4 *>(rp + ((rot + k) & 7) * 16) = buf[m][k];
        }
    }
}

// phi_tile (elu + 1, no weights) as a loop that is not unrolled, for nt threads
// given at run time: one unit (16 independent packed phi pairs) per trip.  The
// code is a few hundred bytes, so a kernel that runs it a few times per launch
// fetches it once; the unrolled form is several kilobytes per call site, each
// run from a cold instruction cache.
template <int D>
__device__ __forceinline__ void phi_tile_rolled(uint8_t *tile, int t, int nt, int valid)
{
    constexpr int kUnits = 128 * (D / 32);
#pragma unroll 1
    for (int u = t; u < kUnits; u += nt) {
        const int row = u & 127, hb = u >> 7;
        uint8_t *rp = tile + (hb >> 1) * kBox + row * 128;
        const int rot = row + (hb & 1) * 4;
        uint4 x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = *reinterpret_cast<const uint4 *>(rp + ((rot + k) & 7) * 16);
        const bool live = row < valid;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            x[k] = live ? make_uint4(phi2(x[k].x), phi2(x[k].y), phi2(x[k].z), phi2(x[k].w)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4 *>(rp + ((rot + k) & 7) * 16) = x[k];
    }
}

// phi of two bf16 values in fp32, split into bf16 high parts (returned) and the
// bf16 rounding of the remainders (*lo): hi + lo carries phi to about 2^-17.
__device__ __forceinline__ uint32_t phi2_split(uint32_t w, uint32_t *lo)
{
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&w);
    const float a = __bfloat162float(x.x), b = __bfloat162float(x.y);
    const float pa = a > 0.f ? a + 1.f : __expf(a), pb = b > 0.f ? b + 1.f : __expf(b);
    const __nv_bfloat16 ha = __float2bfloat16_rn(pa), hb = __float2bfloat16_rn(pb);
    const __nv_bfloat162 l = __floats2bfloat162_rn(pa - __bfloat162float(ha), pb - __bfloat162float(hb));
    *lo = *reinterpret_cast<const uint32_t *>(&l);
    const __nv_bfloat162 h = __halves2bfloat162(ha, hb);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// As phi_tile, with phi split: the high parts in place, the low parts at the
// same offsets of `lo` (a tile of the same layout).
template <int D, int NT>
__device__ __forceinline__ void phi_tile_split(uint8_t *tile, uint8_t *lo, int t, int valid)
{
    constexpr int kUnits = 128 * (D / 32);
    constexpr int NU = (kUnits + NT - 1) / NT;
#pragma unroll 1
    for (int m = 0; m < NU; ++m) {
        const int u = t + NT * m, row = u & 127, hb = u >> 7;
        if (u >= kUnits) break;
        const uint32_t off = (hb >> 1) * kBox + row * 128;
        const int rot = row + (hb & 1) * 4;
        uint4 x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = *reinterpret_cast<const uint4 *>(tile + off + ((rot + k) & 7) * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 h = make_uint4(0u, 0u, 0u, 0u), l = make_uint4(0u, 0u, 0u, 0u);
            if (row < valid) {
                h.x = phi2_split(x[k].x, &l.x);
                h.y = phi2_split(x[k].y, &l.y);
                h.z = phi2_split(x[k].z, &l.z);
                h.w = phi2_split(x[k].w, &l.w);
            }
            *reinterpret_cast<uint4 *>(tile + off + ((rot + k) & 7) * 16) = h;
            *reinterpret_cast<uint4 *>(lo + off + ((rot + k) & 7) * 16) = l;
        }
    }
}

// Descriptor helpers (see la_sm100.cuh for the layouts).
__device__ __forceinline__ uint64_t kmajor(uint32_t tile, int kk)
{
    return desc_sw128(tile + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor(uint32_t tile, int kk, uint32_t lbo)
{
    return desc_sw128(tile + kk * 2048, lbo, 1024);
}
__device__ __forceinline__ uint64_t wdesc(uint32_t w, int kk)
{
    return desc_sw128(w + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048);
}

// Row i of the bf16 state copy (32 columns from col0), MN-major 128-byte swizzled:
// 64-column blocks of D rows x 128 bytes.
template <int D>
__device__ __forceinline__ void put_sb(uint8_t *sb, int i, int col0, const float (&x)[32])
{
#pragma unroll
    for (int c8 = 0; c8 < 32; c8 += 8) {
        const int col = col0 + c8;
        const uint32_t off = (col >> 6) * (D * 128) + i * 128 + ((((col & 63) >> 3) ^ (i & 7)) << 4);
        *reinterpret_cast<uint4 *>(sb + off) =
            make_uint4(pack_bf16(x[c8], x[c8 + 1]), pack_bf16(x[c8 + 2], x[c8 + 3]),
                       pack_bf16(x[c8 + 4], x[c8 + 5]), pack_bf16(x[c8 + 6], x[c8 + 7]));
    }
}
// z_i split into a high and a low bf16 part: rows 1 and 2 of W.
__device__ __forceinline__ void put_z(uint8_t *w, int i, float zv)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
    const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
    uint8_t *blk = w + (i >> 6) * 1024;
    *reinterpret_cast<__nv_bfloat16 *>(blk + sw128_offset(1, i & 63)) = hi;
    *reinterpret_cast<__nv_bfloat16 *>(blk + sw128_offset(2, i & 63)) = lo;
}
// Published scan states use a thread-major layout, so that the 32 rows a warp
// handles are contiguous: the float4 holding columns 4c..4c+3 of row i is at
// float4 index c*D + i, and z_i follows at float D*D + i.
template <int D>
__device__ __forceinline__ void add_state(float (&acc)[32], const float *state, int cg0, int i)
{
    const float4 *s4 = reinterpret_cast<const float4 *>(state);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float4 x = __ldcg(s4 + (size_t)(cg0 + e) * D + i);
        acc[4 * e] += x.x; acc[4 * e + 1] += x.y; acc[4 * e + 2] += x.z; acc[4 * e + 3] += x.w;
    }
}
__device__ __forceinline__ void to_floats(const uint32_t *a, float (&x)[32])
{
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(a[e]);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

inline la_status encode_fn(EncodeTiledFn *out)
{
    static std::mutex mu;
    static EncodeTiledFn fn = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void **)&fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return cuda_status(e);
        if (q != cudaDriverEntryPointSuccess || !fn) {
            fn = nullptr;
            return cuda_status(cudaErrorNotSupported);
        }
    }
    *out = fn;
    return LA_OK;
}

// The tensor-map encoder is a driver call: it needs a current context in the
// calling thread, which the runtime binds only when that thread makes its first
// runtime call that uses the device.  A host thread whose first CUDA work is this
// library has none yet: bind the runtime's primary context of the current device
// (once per thread; a thread without a context cannot be capturing a stream).
inline la_status bind_thread_context()
{
    typedef CUresult (*CtxGetFn)(CUcontext *);
    static std::mutex mu;
    static CtxGetFn get = nullptr;
    static thread_local bool bound = false;
    if (bound) return LA_OK;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!get) {
            cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", (void **)&get, 12000,
                                                             cudaEnableDefault, &q);
            if (e != cudaSuccess) return cuda_status(e);
            if (q != cudaDriverEntryPointSuccess || !get) {
                get = nullptr;
                return cuda_status(cudaErrorNotSupported);
            }
        }
    }
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return cuda_status(cudaErrorInvalidValue);
    if (!ctx) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaSetDevice(dev);
        if (e != cudaSuccess) return cuda_status(e);
    }
    bound = true;
    return LA_OK;
}

// [BH, N, D] bf16 as a 3-D tensor (D, N, BH); box = 64 columns x 128 rows, 128-byte swizzle.
inline la_status make_map(CUtensorMap *m, const void *ptr, int BH, int N, int D)
{
    EncodeTiledFn enc;
    la_status st = encode_fn(&enc);
    if (st == LA_OK) st = bind_thread_context();
    if (st != LA_OK) return st;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LA_OK : cuda_status(cudaErrorInvalidValue);
}

// Programmatic stream serialization is requested only on streams the caller
// created: the default streams (legacy, per-thread) synchronise implicitly with
// other work, and there the kernels launch plainly (their griddepcontrol
// instructions are then no-ops).
inline bool dependent_launch_allowed(cudaStream_t s)
{
    return s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread;
}

// Launches a tensor-core kernel with programmatic stream serialization: its CTAs
// may start (set-up, TMEM allocation) while the previous kernel on the stream
// finishes; the kernel executes griddep_wait() before its first access to global
// memory that an earlier launch may still write (inputs, flags, workspace).
template <typename... Params, typename... Args>
inline la_status launch_dependent(void (*kern)(Params...), unsigned grid, int threads, int smem, cudaStream_t s,
                                  Args... args)
{
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3((unsigned)threads);
    lc.dynamicSmemBytes = (size_t)smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = dependent_launch_allowed(s) ? 1 : 0;
    return cuda_status(cudaLaunchKernelEx(&lc, kern, args...));
}

inline int sm_count()
{
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
    cache[dev] = n;
    return n;
}

}  // namespace tc
}  // namespace la
