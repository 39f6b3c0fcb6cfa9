// FAVOR+ positive random features ("Linear Attention -- Math + Variants",
// Performer: phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m) for r = 0..m-1, whose
// inner products estimate the softmax kernel exp(q . k) without bias; the
// projections w_r (the rows of W [m, d]) are drawn by the caller, orthogonal
// blocks or plain Gaussian rows alike).
//
// x W^T is a dense contraction, so for bf16 with d, m in {64, 128} it runs on
// the tensor cores: a persistent kernel with W resident in shared memory (loaded
// by TMA with the first tile), 128-row tiles of x brought in by TMA, one
// tcgen05.mma group per tile into a TMEM accumulator (two buffers), and two sets
// of epilogue warps, one per accumulator, that take alternate tiles: each adds the
// norm term, takes the exponential with the 1/sqrt(m) scale folded into its
// exponent and stores bf16 rows by TMA.  Other shapes and fp32 run on the CUDA
// cores in fp32.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "la_common.cuh"
#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tc;

static __device__ unsigned g_favor_status;

constexpr float kLog2e = 1.4426950408889634f;
// warp 0: TMA loads, warp 1: MMA issue, warps 2-5: epilogue set 0 (even tiles,
// accumulator 0), warps 6-9: epilogue set 1 (odd tiles, accumulator 1)
constexpr int kFavorThreads = 320;
constexpr uint32_t kOutRows = 32;                 // rows per epilogue warp and per TMA store box
constexpr uint32_t kOutBox = kOutRows * 128;      // [32 rows x 64 bf16] swizzled: 4 KB
constexpr uint64_t kDrainLimitNs = 100000000ull;  // 0.1 s for copies still in flight after an abort

template <int D, int M>
struct FavorCfg {
    static constexpr int kStages = D == 128 ? 3 : 4;
    static constexpr uint32_t kXTile = (D / 64) * kBox;          // one 128-row tile of x
    static constexpr uint32_t kWarpOut = (M / 64) * kOutBox;     // 32 rows of phi: one warp's buffer
    static constexpr uint32_t kWBytes = (D / 64) * M * 128;      // W as D/64 boxes of M rows
    static constexpr uint32_t kOffW = kStages * kXTile;          // W: D/64 boxes of up to 128 rows
    static constexpr uint32_t kOffOut = kOffW + (D / 64) * kBox;  // 8 epilogue warps x 1 buffer
    static constexpr uint32_t kOffBar = kOffOut + 8 * kWarpOut;
    static constexpr uint32_t kSmem = kOffBar + 256;
    static constexpr uint32_t kTmemCols = 2 * M;                 // two accumulators of M columns
    // exponent offset of the 1/sqrt(m) scale: -log2(m) / 2
    static constexpr float kScaleExp = M == 64 ? -3.0f : -3.5f;
    static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct FavorBars {
    uint64_t full[4], empty[4], acc_full[2], acc_free[2];
    uint32_t tmem_base;
    int abort;
};

struct FavorParams {
    int BH, N, nch;
    int T1;     // tiles of one tensor: BH * nch
    int total;  // tiles of the launch: T1 or 2 * T1 (q and k)
};

__device__ __forceinline__ bool fwait(int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return tc::wait_bar(&g_favor_status, abort_flag, bar, parity);
}
__device__ __forceinline__ bool fwait_warp(int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return tc::wait_bar_warp(&g_favor_status, abort_flag, bar, parity);
}

// Tile idx of the launch -> tensor (0: q, 1: k), sequence bh, chunk c.
__device__ __forceinline__ void tile_coords(const FavorParams &p, int idx, int &which, int &bh, int &c)
{
    which = idx >= p.T1;
    const int r = idx - which * p.T1;
    bh = r / p.nch;
    c = r - bh * p.nch;
}

template <int D, int M>
__global__ void __launch_bounds__(kFavorThreads, 1)
favor_tc_kernel(const __grid_constant__ CUtensorMap map_xq, const __grid_constant__ CUtensorMap map_xk,
                const __grid_constant__ CUtensorMap map_oq, const __grid_constant__ CUtensorMap map_ok,
                const __grid_constant__ CUtensorMap map_w, const FavorParams prm)
{
    using CF = FavorCfg<D, M>;
    constexpr int S = CF::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // layout assumption of the swizzled tiles
        if (threadIdx.x == 0) atomicOr(&g_favor_status, kStatusTimeout);
        return;
    }
    FavorBars &bars = *reinterpret_cast<FavorBars *>(smem_raw + CF::kOffBar);
    uint8_t *xs = smem_raw;
    uint8_t *ws = smem_raw + CF::kOffW;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    griddep_launch_dependents();

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 4);  // one arrival per epilogue warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.acc_full[b], 1);
            mbar_init(&bars.acc_free[b], 4);
        }
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars.tmem_base, CF::kTmemCols);
        tmem_relinquish();
    }
    griddep_wait();  // W and x may be written by the launch before this one
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    int *abort_flag = &bars.abort;
    const int ntiles =
        (int)blockIdx.x < prm.total ? (prm.total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA loads
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int s = j % S;
                if (j >= S && !fwait(abort_flag, &bars.empty[s], ((j / S) - 1) & 1)) break;
                int which, bh, c;
                tile_coords(prm, (int)blockIdx.x + j * (int)gridDim.x, which, bh, c);
                if (j == 0) {
                    // W [M, D] rides on the first tile's barrier: K-major swizzled B operand,
                    // box b holding columns 64b .. 64b + 63 of all M rows
                    mbar_arrive_expect_tx(&bars.full[0], CF::kXTile + CF::kWBytes);
#pragma unroll
                    for (int bx = 0; bx < D / 64; ++bx)
                        tma_load_3d(ws + bx * kBox, &map_w, &bars.full[0], 64 * bx, 0, 0);
                } else {
                    mbar_arrive_expect_tx(&bars.full[s], CF::kXTile);
                }
#pragma unroll
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load_3d_hint(xs + s * CF::kXTile + bx * kBox, which ? &map_xk : &map_xq, &bars.full[s],
                                     64 * bx, c * 128, bh, pol);
                ++issued;
            }
            // after an abort, let the loads still in flight land before the CTA exits
            for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
                (void)mbar_wait(&bars.full[j % S], (j / S) & 1, kDrainLimitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, M, false, false);  // x W^T, both K-major
            const uint32_t xa = smem_u32(xs), wa = smem_u32(ws);
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int s = j % S, b = j & 1;
                if (!fwait(abort_flag, &bars.full[s], (j / S) & 1)) break;
                if (j >= 2 && !fwait(abort_flag, &bars.acc_free[b], ((j >> 1) - 1) & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + b * M, kmajor(xa + s * CF::kXTile, kk), kmajor(wa, kk), idesc, kk > 0 ? 1u : 0u);
                mma_commit(&bars.acc_full[b]);
                ++issued;
            }
            if (issued > 0)  // the last MMAs have finished with TMEM before it is freed
                (void)mbar_wait(&bars.acc_full[(issued - 1) & 1], ((issued - 1) >> 1) & 1, kDrainLimitNs);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int qw = warp & 3;             // TMEM lane quarter this warp may access
        const int set = (warp - 2) >> 2;     // tiles j with j % 2 == set, accumulator `set`
        const int i = qw * 32 + lane;        // row of the tile
        const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
        uint8_t *ob = smem_raw + CF::kOffOut + (warp - 2) * CF::kWarpOut;
        const uint64_t pol = l2_policy_evict_first();
        for (int j = set; j < ntiles; j += 2) {
            const int s = j % S, b = j & 1;
            int which, bh, c;
            tile_coords(prm, (int)blockIdx.x + j * (int)gridDim.x, which, bh, c);
            // |x_i|^2 from the staged tile (rows past the sequence were zero-filled)
            if (!fwait_warp(abort_flag, &bars.full[s], (j / S) & 1)) break;
            float nrm = 0.f;
            const uint8_t *xt = xs + s * CF::kXTile;
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    // the swizzle permutes 16-byte chunks within the row: any order covers it
                    const uint4 w4 = *reinterpret_cast<const uint4 *>(xt + bx * kBox + i * 128 + (((u + i) & 7) << 4));
                    const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv[e]));
                        nrm = fmaf(f.x, f.x, nrm);
                        nrm = fmaf(f.y, f.y, nrm);
                    }
                }
            }
            if (!fwait_warp(abort_flag, &bars.acc_full[b], (j >> 1) & 1)) break;
            tc_fence_after();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.empty[s]);  // the MMAs and this warp are done with x
            // phi = 2^(acc log2(e) - |x|^2 log2(e) / 2 - log2(m) / 2)
            const float cexp = fmaf(-0.5f * kLog2e, nrm, CF::kScaleExp);
            // this warp's store of two tiles ago has finished reading the buffer
            if (lane == 0) tma_store_wait_read_all();
            __syncwarp();
#pragma unroll 1
            for (int cc = 0; cc < M / 64; ++cc) {
                uint32_t v[64];
                tmem_ld32(tl + b * M + cc * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(tl + b * M + cc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tmem_ld_wait();
                uint8_t *rowp = ob + cc * kOutBox + lane * 128;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = exp2f(fmaf(__uint_as_float(v[8 * u + e]), kLog2e, cexp));
                    *reinterpret_cast<uint4 *>(rowp + ((u ^ (lane & 7)) << 4)) =
                        make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                                   pack_bf16(f[6], f[7]));
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars.acc_free[b]);
                // rows past the end of the sequence fall outside the tensor and are not
                // written; a box that starts past the end is not issued at all
                if (c * 128 + qw * 32 < prm.N) {
#pragma unroll
                    for (int cc = 0; cc < M / 64; ++cc)
                        tma_store_3d_hint(which ? &map_ok : &map_oq, ob + cc * kOutBox, 64 * cc, c * 128 + qw * 32,
                                          bh, pol);
                }
                tma_store_commit();
            }
        }
        if (lane == 0) tma_store_wait_all();  // every store complete before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, CF::kTmemCols);
}

// [BH, N, D] bf16 as a 3-D tensor (D, N, BH) with a box of 64 columns x `rows` rows.
la_status make_map_rows(CUtensorMap *m, const void *ptr, int BH, int N, int D, int rows)
{
    EncodeTiledFn enc;
    la_status st = encode_fn(&enc);
    if (st == LA_OK) st = bind_thread_context();
    if (st != LA_OK) return st;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LA_OK : cuda_status(cudaErrorInvalidValue);
}

template <int D, int M>
la_status launch_tc(const void *xq, const void *xk, const void *W, void *oq, void *ok, int BH, int N,
                    cudaStream_t stream)
{
    using CF = FavorCfg<D, M>;
    CUtensorMap mxq, mxk, moq, mok, mw;
    la_status st;
    if ((st = make_map_rows(&mxq, xq, BH, N, D, 128)) != LA_OK) return st;
    if ((st = make_map_rows(&mxk, xk ? xk : xq, BH, N, D, 128)) != LA_OK) return st;
    if ((st = make_map_rows(&moq, oq, BH, N, M, (int)kOutRows)) != LA_OK) return st;
    if ((st = make_map_rows(&mok, ok ? ok : oq, BH, N, M, (int)kOutRows)) != LA_OK) return st;
    if ((st = make_map_rows(&mw, W, 1, M, D, M)) != LA_OK) return st;
    FavorParams prm;
    prm.BH = BH;
    prm.N = N;
    prm.nch = ceil_div(N, 128);
    prm.T1 = BH * prm.nch;
    prm.total = xk ? 2 * prm.T1 : prm.T1;
    if ((st = ensure_smem((const void *)favor_tc_kernel<D, M>, (int)CF::kSmem)) != LA_OK) return st;
    const int grid = prm.total < sm_count() ? prm.total : sm_count();
    st = launch_dependent(favor_tc_kernel<D, M>, (unsigned)grid, kFavorThreads, (int)CF::kSmem, stream, mxq, mxk,
                          moq, mok, mw, prm);
    count_launches();
    return st;
}

// ---------------------------------------------------------------- CUDA cores
constexpr int kSimtThreads = 256;
constexpr int kSimtRows = 8;  // rows of x per block iteration

// Block: W [m, d] in shared memory as fp32 (rows padded to d + 1 so that the
// lanes of a warp, which take consecutive features r, read different banks);
// then groups of 8 rows of x: their squared norms, and every feature of every row.
template <typename T>
__global__ void __launch_bounds__(kSimtThreads)
favor_simt_kernel(const T *__restrict__ xq, const T *__restrict__ xk, const T *__restrict__ W, T *__restrict__ oq,
                  T *__restrict__ ok, long long rows, int d, int m, float inv_sqrt_m, int tensors)
{
    extern __shared__ float fsm[];
    float *wsm = fsm;                       // [m][d + 1]
    float *xsm = wsm + m * (d + 1);         // [kSimtRows][d]
    float *nsm = xsm + kSimtRows * d;       // [kSimtRows]
    for (int e = threadIdx.x; e < m * d; e += kSimtThreads)
        wsm[(e / d) * (d + 1) + e % d] = Elem<T>::to_f32(W[e]);
    const long long groups = (rows + kSimtRows - 1) / kSimtRows, total = groups * tensors;
    for (long long g = blockIdx.x; g < total; g += gridDim.x) {
        const int which = g >= groups;
        const long long r0 = (g - which * groups) * kSimtRows;
        const T *x = which ? xk : xq;
        T *o = which ? ok : oq;
        __syncthreads();  // W is in place; the previous group's rows are no longer read
        for (int e = threadIdx.x; e < kSimtRows * d; e += kSimtThreads) {
            const long long r = r0 + e / d;
            xsm[e] = r < rows ? Elem<T>::to_f32(x[r * d + e % d]) : 0.f;
        }
        __syncthreads();
        if (threadIdx.x < kSimtRows) {
            float s = 0.f;
            for (int c = 0; c < d; ++c) s = fmaf(xsm[threadIdx.x * d + c], xsm[threadIdx.x * d + c], s);
            nsm[threadIdx.x] = s;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kSimtRows * m; e += kSimtThreads) {
            const int rr = e / m, f = e - rr * m;
            if (r0 + rr >= rows) break;  // e only grows: later rows are past the end too
            const float *xr = xsm + rr * d, *wr = wsm + f * (d + 1);
            float dot = 0.f;
            for (int c = 0; c < d; ++c) dot = fmaf(xr[c], wr[c], dot);
            o[(r0 + rr) * m + f] = Elem<T>::from_f32(expf(dot - 0.5f * nsm[rr]) * inv_sqrt_m);
        }
    }
}

template <typename T>
la_status launch_simt(const void *xq, const void *xk, const void *W, void *oq, void *ok, long long rows, int d,
                      int m, cudaStream_t stream)
{
    const int smem = (int)sizeof(float) * (m * (d + 1) + kSimtRows * d + kSimtRows);
    // The attribute is set once, to the size of the largest shape (d = m = 128), so
    // that launches of every size fit it whatever order they come in.
    constexpr int kMaxSmem = (int)sizeof(float) * (128 * 129 + kSimtRows * 128 + kSimtRows);
    la_status st = ensure_smem((const void *)favor_simt_kernel<T>, kMaxSmem);
    if (st != LA_OK) return st;
    const int tensors = xk ? 2 : 1;
    const long long total = (rows + kSimtRows - 1) / kSimtRows * tensors;
    const long long cap = 4LL * tc::sm_count();
    const int grid = (int)(total < cap ? total : cap);
    const float inv_sqrt_m = (float)(1.0 / sqrt((double)m));
    favor_simt_kernel<T><<<grid, kSimtThreads, smem, stream>>>((const T *)xq, (const T *)xk, (const T *)W, (T *)oq,
                                                               (T *)ok, rows, d, m, inv_sqrt_m, tensors);
    count_launches();
    return cuda_status(cudaGetLastError());
}

}  // namespace

la_status favor_features(const void *xq, const void *xk, const void *W, void *oq, void *ok, int BH, int N, int d,
                         int m, la_dtype dtype, cudaStream_t stream)
{
    // (sequences shorter than one 128-row tile, whose tile would be taller than the
    // tensor, stay on the CUDA cores, as in the attention kernels)
    if (dtype == LA_BF16 && (d == 64 || d == 128) && (m == 64 || m == 128) && N >= 128) {
        if (d == 64)
            return m == 64 ? launch_tc<64, 64>(xq, xk, W, oq, ok, BH, N, stream)
                           : launch_tc<64, 128>(xq, xk, W, oq, ok, BH, N, stream);
        return m == 64 ? launch_tc<128, 64>(xq, xk, W, oq, ok, BH, N, stream)
                       : launch_tc<128, 128>(xq, xk, W, oq, ok, BH, N, stream);
    }
    const long long rows = (long long)BH * N;
    return dtype == LA_F32 ? launch_simt<float>(xq, xk, W, oq, ok, rows, d, m, stream)
                           : launch_simt<__nv_bfloat16>(xq, xk, W, oq, ok, rows, d, m, stream);
}

la_status favor_read_status(cudaStream_t s, unsigned *bits)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_favor_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_favor_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // namespace la
