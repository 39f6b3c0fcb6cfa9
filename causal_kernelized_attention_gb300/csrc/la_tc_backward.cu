// Backward pass of the causal form on the tensor cores: bf16 q, k, v, dO, dk = dv = 64
// (narrower widths on the same tiles: see backward_tc_eligible), N >= 128; fp32 accumulation, bf16 gradients.  The same chain rule as the CUDA-core
// backward in la_backward.cu (the pages give no gradient; "Linear Attention -- Math +
// Variants", Chunkwise parallelism: training runs the chunked form), over chunks of
// C = 128 tokens, with every block product a tcgen05 MMA:
//
//   1. chunk states     A_c = phi(K_c)^T [V_c | 1]                        -> buf[c]
//   2. forward scan     buf[c] = sum_{c' < c} A_c' = [S | z] before chunk c
//   3. dq, per chunk    T = phi(Q) phi(K)^T, P = bf16(tril T)             (TMEM)
//                       [num | den] = P [V | 1] + phi(Q) [S | z]
//                       d = max(den, eps), dN = dO / d, dd = -(dO . num / d) / d (0 if clamped)
//                       U = dN V^T, U' = bf16(tril(U + dd 1^T))           (TMEM)
//                       dphi(Q) = U' phi(K) + dN S^T (+ dd z^T, fp32)  ->  dq = dphi(Q) phi'(q)
//                       B_c = phi(Q)^T [dN | dd]                          -> buf[c]
//                       dN (bf16) and dd (fp32) to scratch for step 5
//   4. reverse scan     buf[c] = sum_{c' > c} B_c' = [R | r] after chunk c
//   5. dk, dv per chunk T^T = phi(K) phi(Q)^T, P^T = bf16(triu T^T)       (TMEM)
//                       U^T = V dN^T, U'^T = bf16(triu(U^T + 1 dd^T))     (TMEM)
//                       dV = P^T dN + phi(K) R
//                       dphi(K) = U'^T phi(Q) + V R^T (+ 1 r^T, fp32)  ->  dk = dphi(K) phi'(k)
//
// Operands: the Q, K, V, dO and dN tiles are [128 tokens x 64] bf16 boxes, 128-byte
// swizzled (TMA); a tile serves as a K-major operand (tokens as rows, features
// contiguous) and as an MN-major one (tokens as the K index) without a copy, and the
// bf16 image of a state [f][v] (values contiguous) serves as the MN-major B of
// phi(Q) S and phi(K) R and as the K-major B of dN S^T and V R^T.  P, U', P^T and
// U'^T are formed in TMEM by the epilogue threads over the fp32 products and read
// by the next MMAs from there.  The extra N columns of the fused products live in
// one 128 x 128-byte block: column 0 of each row is 1 (the row sums P 1), the third
// 16-byte chunk holds dd (the r column of B_c), the fifth z as a bf16 high + low pair
// (the denominator's phi(Q) z), each reached through the descriptor's LBO.
//
// One CTA per chunk (grid = heads x chunks): 320 threads, two groups of four
// epilogue warps (each covering the four TMEM lane quadrants), a TMA warp and an
// MMA warp; 256 TMEM columns and about 105 KB (dq) or 74 KB (dk, dv) of shared
// memory, so two CTAs share an SM.  Every wait is bounded; on expiry the CTA
// records LA_ERR_TIMEOUT in this file's status word and winds down.
#include "la_common.cuh"
#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"
#include "la_tc_pad.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tc;

static __device__ unsigned g_bw_status;

constexpr int D = 64;
constexpr uint32_t kTile = kC * D * 2;  // one [128 x 64] bf16 tile: 16 KB
constexpr uint32_t kImg = D * D * 2;    // a state image [64 x 64] bf16: 8 KB
constexpr int kE = D * (D + 1);         // floats per chunk state
constexpr int kThreads = 320;           // warps 0-7 epilogue groups, 8 TMA, 9 MMA
constexpr int kWork = 256;
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kOnesOff = 0, kDdOff = 32, kZOff = 64;  // byte offsets of the extra columns' chunks
constexpr uint64_t kDrainNs = 100000000ull;

// State layout in buf (fp32, kE floats per chunk): the float4 of columns 4e..4e+3 of
// row f at float4 index e * D + f; z_f (or r_f) at float D * D + f.  A thread per row
// reads and writes whole float4s and a warp's 32 rows are contiguous.

__device__ __forceinline__ bool wait_b(int *abort_flag, uint64_t *bar)
{
    return wait_bar(&g_bw_status, abort_flag, bar, 0);
}
__device__ __forceinline__ bool wait_w(int *abort_flag, uint64_t *bar)
{
    return wait_bar_warp(&g_bw_status, abort_flag, bar, 0);
}
__device__ __forceinline__ void drain(uint64_t *bar)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, 0) && globaltimer_ns() - t0 < kDrainNs) {
    }
}

// Row f, columns [c0, c0 + 16) of a bf16 image [64 x 64] (128-byte swizzled rows).
__device__ __forceinline__ void put_img16(uint8_t *img, int f, int c0, const float (&x)[16])
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int col = c0 + 8 * h;
        *reinterpret_cast<uint4 *>(img + f * 128 + (((col >> 3) ^ (f & 7)) << 4)) =
            make_uint4(pack_bf16(x[8 * h], x[8 * h + 1]), pack_bf16(x[8 * h + 2], x[8 * h + 3]),
                       pack_bf16(x[8 * h + 4], x[8 * h + 5]), pack_bf16(x[8 * h + 6], x[8 * h + 7]));
    }
}
// The 16-byte chunk at byte offset `off` (0, 32 or 64) of row r of the extra-column
// block, with the pair (a, b) in its first two columns and zeros after.
__device__ __forceinline__ void put_extra(uint8_t *blk, int r, uint32_t off, uint32_t pair)
{
    *reinterpret_cast<uint4 *>(blk + r * 128 + ((((off >> 4)) ^ (r & 7)) << 4)) = make_uint4(pair, 0u, 0u, 0u);
}
// The extra-column block's constant part: column 0 = 1, every other chunk zero
// except those at kDdOff and kZOff, which their writers fill.
__device__ __forceinline__ void init_extra(uint8_t *blk, int t, int nt)
{
    for (int u = t; u < kC * 8; u += nt) {
        const int r = u >> 3, ch = u & 7;  // physical chunk ch of row r
        const int logical = ch ^ (r & 7);
        if (logical == (int)(kDdOff >> 4) || logical == (int)(kZOff >> 4)) continue;
        const uint32_t x = logical == 0 ? 0x3F80u : 0u;
        *reinterpret_cast<uint4 *>(blk + r * 128 + ch * 16) = make_uint4(x, 0u, 0u, 0u);
    }
}
// A chunk state, copied from buf into shared memory (the S part at st in buf's layout,
// the last column at zs), into a bf16 image: load_state (thread t of 256: row f =
// t % 64, columns 16 (t / 64) .. and, for t < 64, the last column) and put_state (the
// image row part; the fp32 last column to zf[] and, if zblk, as a hi + lo pair into
// the extra-column block, rows 0..63).
__device__ __forceinline__ void load_state(const float *st, const float *zs, int t, float (&x)[16], float &z)
{
    const int f = t & 63, cg = t >> 6;
    const float4 *s4 = reinterpret_cast<const float4 *>(st);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float4 a = s4[(4 * cg + e) * D + f];
        x[4 * e] = a.x; x[4 * e + 1] = a.y; x[4 * e + 2] = a.z; x[4 * e + 3] = a.w;
    }
    z = cg == 0 ? zs[f] : 0.f;
}
__device__ __forceinline__ void put_state(uint8_t *img, float *zf, uint8_t *zblk, int t, const float (&x)[16], float z)
{
    const int f = t & 63, cg = t >> 6;
    put_img16(img, f, 16 * cg, x);
    if (cg == 0) {
        zf[f] = z;
        if (zblk) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(z);
            const __nv_bfloat16 lo = __float2bfloat16_rn(z - __bfloat162float(hi));
            const __nv_bfloat162 pr = __halves2bfloat162(hi, lo);
            put_extra(zblk, f, kZOff, *reinterpret_cast<const uint32_t *>(&pr));
        }
    }
}

// Row 32 q + lane of a 128 x 128 fp32 product at TMEM address tb (this warp's lane
// quadrant), plus bias(col), masked (kLower: col <= row; else col >= row) and rounded
// to bf16, written back packed over columns 0..63 (pairs of columns per 32-bit
// column: the A operand layout of a TMEM-sourced MMA).  Key block kb (32 columns) is
// read in two halves; the packed half-block it produces lands on columns already read.
template <bool kLower, typename Bias>
__device__ __forceinline__ void tmem_mask_bf16(uint32_t tb, int q, int lane, Bias bias)
{
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        const bool any = kLower ? kb <= q : kb >= q;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t pk[8];
            if (any) {
                uint32_t t[16];
                tmem_ld16(tb + kb * 32 + 16 * hb, t);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = 16 * hb + 2 * e;  // column within the block
                    const int c = kb * 32 + j;
                    const bool k0 = kb != q || (kLower ? j <= lane : j >= lane);
                    const bool k1 = kb != q || (kLower ? j + 1 <= lane : j + 1 >= lane);
                    pk[e] = pack_bf16(k0 ? __uint_as_float(t[2 * e]) + bias(c) : 0.f,
                                      k1 ? __uint_as_float(t[2 * e + 1]) + bias(c + 1) : 0.f);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) pk[e] = 0u;
            }
            tmem_st8(tb + kb * 16 + 8 * hb, pk);
        }
    }
    tmem_st_wait();
}

// As tmem_mask_bf16 (lower mask), split between two groups of warps on the same
// rows: group g converts key blocks 2g, 2g + 1; every thread reads its blocks into
// registers before either group writes (the packed output of blocks 2, 3 lands on
// block 1's columns), with one barrier of both groups (bar_id, 256 threads) between.
// Every thread of both groups calls it; with live == false it only takes part in the
// barrier (so that a CTA winding down after a failed wait cannot stall there).
template <typename Bias>
__device__ __forceinline__ void tmem_tril_bf16_split(bool live, uint32_t tb, int q, int lane, int g, uint32_t bar_id,
                                                     Bias bias)
{
    uint32_t pk[2][2][8];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int kb = 2 * g + b;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            if (live && kb <= q) {
                uint32_t t[16];
                tmem_ld16(tb + kb * 32 + 16 * hb, t);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = 16 * hb + 2 * e;
                    const int c = kb * 32 + j;
                    const bool k0 = kb != q || j <= lane, k1 = kb != q || j + 1 <= lane;
                    pk[b][hb][e] = pack_bf16(k0 ? __uint_as_float(t[2 * e]) + bias(c) : 0.f,
                                             k1 ? __uint_as_float(t[2 * e + 1]) + bias(c + 1) : 0.f);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) pk[b][hb][e] = 0u;
            }
        }
    }
    named_bar_sync(bar_id, 256);
    if (!live) return;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int kb = 2 * g + b;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) tmem_st8(tb + kb * 16 + 8 * hb, pk[b][hb]);
    }
    tmem_st_wait();
}

// 16 bf16 values of row r, columns [c0, c0 + 16), of a 128-byte swizzled tile.
__device__ __forceinline__ void ld_row16(const uint8_t *tile, int r, int c0, float (&x)[16])
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 u = *reinterpret_cast<const uint4 *>(tile + r * 128 + ((((c0 >> 3) + h) ^ (r & 7)) << 4));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[e]);
            x[8 * h + 2 * e] = __bfloat162float(b.x);
            x[8 * h + 2 * e + 1] = __bfloat162float(b.y);
        }
    }
}
__device__ __forceinline__ void st_row16(uint8_t *tile, int r, int c0, const float (&x)[16])
{
#pragma unroll
    for (int h = 0; h < 2; ++h)
        *reinterpret_cast<uint4 *>(tile + r * 128 + ((((c0 >> 3) + h) ^ (r & 7)) << 4)) =
            make_uint4(pack_bf16(x[8 * h], x[8 * h + 1]), pack_bf16(x[8 * h + 2], x[8 * h + 3]),
                       pack_bf16(x[8 * h + 4], x[8 * h + 5]), pack_bf16(x[8 * h + 6], x[8 * h + 7]));
}
// phi'(x) from phi(x) for elu + 1: 1 where x > 0 (phi > 1), exp(x) = phi(x) otherwise.
__device__ __forceinline__ float dphi(float phi) { return fminf(phi, 1.f); }

struct Params {
    int N, BH, nC;
    float eps;
    int dk;  // q, k, dq, dk width (at most D; columns past it are zero in phi(K), clipped from the stores)
};

// ---------------------------------------------------------------------- 1. chunk states
struct StateSmem {
    uint8_t k[kTile];
    uint8_t v[kTile];
    uint8_t extra[kC * 128];
    uint64_t k_full, full, mma;  // k_full: K landed; full: V landed
    uint32_t tmem_base;
    int abort;
};

constexpr int kStateThreads = 256;

__global__ void __launch_bounds__(kStateThreads)
bwd_tc_state(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v, float *buf,
             const Params prm)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    StateSmem &sm = *reinterpret_cast<StateSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = (int)blockIdx.x / prm.nC, c = (int)blockIdx.x % prm.nC;
    if (tid == 0) {
        mbar_init(&sm.k_full, 1);
        mbar_init(&sm.full, 1);
        mbar_init(&sm.mma, 1);
        sm.abort = (smem_u32(smem_raw) & 1023u) == 0 ? 0 : 1;
        if (sm.abort) atomicOr(&g_bw_status, kStatusTimeout);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 128);
        tmem_relinquish();
    }
    init_extra(sm.extra, tid, kStateThreads);
    if (tid < kC) put_extra(sm.extra, tid, kDdOff, 0u);  // no dd or z here
    if (tid < kC) put_extra(sm.extra, tid, kZOff, 0u);
    if (tid == 32) {  // into L2 while an earlier kernel on the stream finishes (the L2 is coherent)
        tma_prefetch_3d(&map_k, 0, c * kC, bh);
        tma_prefetch_3d(&map_v, 0, c * kC, bh);
    }
    griddep_wait();
    griddep_launch_dependents();  // after the wait: see the dq kernel
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    int *abort_flag = &sm.abort;
    bool loaded = false;
    if (tid == 0 && !aborted(abort_flag)) {
        const uint64_t pol = l2_policy_evict_last();  // read again by the dq and dk, dv kernels
        mbar_arrive_expect_tx(&sm.k_full, kTile);
        tma_load_3d_hint(sm.k, &map_k, &sm.k_full, 0, c * kC, bh, pol);
        mbar_arrive_expect_tx(&sm.full, kTile);
        tma_load_3d_hint(sm.v, &map_v, &sm.full, 0, c * kC, bh, pol);
        loaded = true;
    }
    bool ok = !aborted(abort_flag) && wait_w(abort_flag, &sm.k_full);
    if (ok) {
        phi_tile_rolled<D>(sm.k, tid, kStateThreads, prm.N - c * kC);
        if (prm.dk < D) zero_cols<D>(sm.k, tid, kStateThreads, prm.dk);
        fence_proxy_async_smem();
        ok = wait_w(abort_flag, &sm.full);
    }
    __syncthreads();
    ok = ok && !aborted(abort_flag);
    bool issued = false;
    if (tid == 0 && ok) {
        issued = true;
        tc_fence_after();
        const uint32_t ka = smem_u32(sm.k), va = smem_u32(sm.v), ex = smem_u32(sm.extra);
        const uint32_t id = idesc_bf16_f32(128, D + 16, true, true);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
            mma_ss(tmem, mnmajor(ka, kk, 0), mnmajor(va, kk, ex + kOnesOff - va), id, kk > 0 ? 1u : 0u);
        mma_commit(&sm.mma);
    }
    if (warp < 2 && ok) {
        ok = wait_w(abort_flag, &sm.mma);
        if (ok) {
            tc_fence_after();
            const int f = 32 * warp + lane;  // rows 0..63 (64..127 repeat them)
            const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
            float4 *out = reinterpret_cast<float4 *>(buf + ((size_t)bh * prm.nC + c) * kE);
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t a[16];
                tmem_ld16(tl + 16 * blk, a);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    out[(4 * blk + e) * D + f] = make_float4(__uint_as_float(a[4 * e]), __uint_as_float(a[4 * e + 1]),
                                                             __uint_as_float(a[4 * e + 2]),
                                                             __uint_as_float(a[4 * e + 3]));
            }
            buf[((size_t)bh * prm.nC + c) * kE + D * D + f] = __uint_as_float(tmem_ld1(tl + D));
            tmem_ld_wait();
        }
    }
    if (tid == 0 && loaded) {
        drain(&sm.k_full);
        drain(&sm.full);
    }
    if (issued) drain(&sm.mma);  // the committed group completes before TMEM is freed
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------- 2., 4. scans
// Exclusive scan over the nC chunk states of every head, in place: prefix (forward)
// or suffix (reverse).  Thread = (head, float4 of the state); every load of a round
// of 16 chunks is issued before the first store.
constexpr int kScanThreads = 256;
__global__ void __launch_bounds__(kScanThreads)
bwd_tc_scan(float *buf, int nC, int BH, int reverse)
{
    constexpr int E4 = kE / 4;
    const long long gidx = (long long)blockIdx.x * kScanThreads + threadIdx.x;
    griddep_wait();
    griddep_launch_dependents();  // after the wait: see the dq kernel
    if (gidx >= (long long)BH * E4) return;
    const long long bh = gidx / E4, e = gidx % E4;
    float4 *p = reinterpret_cast<float4 *>(buf) + bh * (long long)nC * E4 + e;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < nC; i += 16) {
        float4 x[16];
        const int m = min(16, nC - i);
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (u < m) x[u] = __ldcg(p + (long long)(reverse ? nC - 1 - (i + u) : i + u) * E4);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (u < m) {
                __stcg(p + (long long)(reverse ? nC - 1 - (i + u) : i + u) * E4, run);
                run.x += x[u].x; run.y += x[u].y; run.z += x[u].z; run.w += x[u].w;
            }
        }
    }
}

// ---------------------------------------------------------------------- 3. dq
struct DqSmem {
    uint8_t q[kTile];   // phi(Q)
    uint8_t k[kTile];   // phi(K)
    uint8_t v[kTile];
    uint8_t go[kTile];  // dO, then dq staged
    uint8_t dn[kTile];  // the fp32 state S before the chunk as copied, then dN (bf16), also stored to scratch
    uint8_t simg[kImg]; // bf16 S before the chunk, [f][v]
    uint8_t extra[kC * 128];
    float zf[D];        // z before the chunk (fp32)
    float gpart[2][kC]; // each group's half of dO . o per row
    // qk_full: Q, K landed; full: V, dO landed; st_full: the state landed
    uint64_t qk_full, full, st_full, ready, t_full, p_full, o_full, dn_ready, u_full, bc_full, up_full, g_full, dq_staged, drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(DqSmem) + 1024 <= 232448 / 2, "two dq CTAs per SM");
static_assert(kTile == D * D * sizeof(float), "the state's fp32 copy fits the dN tile");

// TMEM of the dq kernel: T at 0 (then P over its first 64 columns), [num | den] at
// 128 (80 columns); after the output epilogue has read them, U at 0 (then U' over
// its first 64 columns), dphi(Q) at 64 and B_c at 128.
constexpr uint32_t tT = 0, tO = 128, tG = 64;

__global__ void __launch_bounds__(kThreads, 2)
bwd_tc_dq(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
          const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
          const __grid_constant__ CUtensorMap map_dn, const __grid_constant__ CUtensorMap map_dq, float *buf,
          float *ddbuf, const Params prm)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    DqSmem &sm = *reinterpret_cast<DqSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = (int)blockIdx.x / prm.nC, c = (int)blockIdx.x % prm.nC;
    const int len = min(kC, prm.N - c * kC);
    float *slot = buf + ((size_t)bh * prm.nC + c) * kE;
    if (tid == 0) {
        uint64_t *bars[] = {&sm.qk_full, &sm.full, &sm.st_full, &sm.t_full, &sm.o_full, &sm.u_full, &sm.bc_full, &sm.g_full, &sm.drain};
        for (uint64_t *b : bars) mbar_init(b, 1);
        mbar_init(&sm.ready, kWork);
        mbar_init(&sm.p_full, kWork);
        mbar_init(&sm.dn_ready, kWork);
        mbar_init(&sm.up_full, kWork);
        mbar_init(&sm.dq_staged, kWork);
        sm.abort = (smem_u32(smem_raw) & 1023u) == 0 ? 0 : 1;
        if (sm.abort) atomicOr(&g_bw_status, kStatusTimeout);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid < kWork) init_extra(sm.extra, tid, kWork);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    int *abort_flag = &sm.abort;

    // Dependent launch.  Every kernel of this backward triggers its dependents only
    // after its own griddep_wait() has returned, so when this grid starts, every grid
    // before the scan that precedes it has completed: q, k, v and dO (none of which
    // the scan writes) are read and phi applied while the scan may still run.  Only
    // the chunk state, which the scan writes, is read after the wait.
    if (warp == kTmaWarp) {
        const bool go = lane == 0 && !aborted(abort_flag);
        if (go) {
            const uint64_t pol = l2_policy_evict_first();
            mbar_arrive_expect_tx(&sm.qk_full, 2 * kTile);  // phi starts on these
            tma_load_3d_hint(sm.q, &map_q, &sm.qk_full, 0, c * kC, bh, pol);
            tma_load_3d_hint(sm.k, &map_k, &sm.qk_full, 0, c * kC, bh, l2_policy_evict_last());
            mbar_arrive_expect_tx(&sm.full, 2 * kTile);
            tma_load_3d_hint(sm.v, &map_v, &sm.full, 0, c * kC, bh, l2_policy_evict_last());
            tma_load_3d_hint(sm.go, &map_do, &sm.full, 0, c * kC, bh, pol);
        }
        griddep_wait();
        griddep_launch_dependents();
        if (go) {
            mbar_arrive_expect_tx(&sm.st_full, (D * D + D) * sizeof(float));
            bulk_load(sm.dn, slot, D * D * sizeof(float), &sm.st_full);
            bulk_load(sm.zf, slot + D * D, D * sizeof(float), &sm.st_full);
            drain(&sm.qk_full);  // no copy may still be writing shared memory when the CTA exits
            drain(&sm.full);
            drain(&sm.st_full);
        }
    } else if (warp == kMmaWarp) {
        griddep_wait();
        griddep_launch_dependents();
        if (lane == 0) {
            const uint32_t qa = smem_u32(sm.q), ka = smem_u32(sm.k), va = smem_u32(sm.v), dna = smem_u32(sm.dn);
            const uint32_t sa = smem_u32(sm.simg), ex = smem_u32(sm.extra);
            bool ok = wait_b(abort_flag, &sm.ready);
            if (ok) {  // T = phi(Q) phi(K)^T
                tc_fence_after();
                const uint32_t id = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + tT, kmajor(qa, kk), kmajor(ka, kk), id, kk > 0);
                mma_commit(&sm.t_full);
            }
            if (ok && (ok = wait_b(abort_flag, &sm.p_full)) && (ok = wait_b(abort_flag, &sm.full))) {
                // [num | den] = P [V | 1] + phi(Q) [S | z]
                tc_fence_after();
                const uint32_t id = idesc_bf16_f32(128, D + 16, false, true);
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_ts(tmem + tO, tmem + tT + kk * 8, mnmajor(va, kk, ex + kOnesOff - va), id, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + tO, kmajor(qa, kk), mnmajor(sa, kk, ex + kZOff - sa), id, 1u);
                mma_commit(&sm.o_full);
            }
            if (ok && (ok = wait_b(abort_flag, &sm.dn_ready))) {
                tc_fence_after();
                {  // U = dN V^T
                    const uint32_t id = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + tT, kmajor(dna, kk), kmajor(va, kk), id, kk > 0);
                    mma_commit(&sm.u_full);
                }
                {  // B_c = phi(Q)^T [dN | dd]: rows 64..127 repeat rows 0..63 (LBO 0); it runs
                   // while the epilogue warps form U'
                    const uint32_t id = idesc_bf16_f32(128, D + 16, true, true);
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_ss(tmem + tO, mnmajor(qa, kk, 0), mnmajor(dna, kk, ex + kDdOff - dna), id, kk > 0);
                    mma_commit(&sm.bc_full);
                }
            }
            if (ok && (ok = wait_b(abort_flag, &sm.up_full))) {  // dphi(Q) = U' phi(K) + dN S^T
                tc_fence_after();
                const uint32_t id1 = idesc_bf16_f32(128, D, false, true);
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) mma_ts(tmem + tG, tmem + tT + kk * 8, mnmajor(ka, kk, 0), id1, kk > 0);
                const uint32_t id2 = idesc_bf16_f32(128, D, false, false);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + tG, kmajor(dna, kk), kmajor(sa, kk), id2, 1u);
                mma_commit(&sm.g_full);
            }
            mma_commit(&sm.drain);  // every MMA issued completes before TMEM is freed
            drain(&sm.drain);
        }
    } else {
        // ---------------------------------------------------------------- warps 0-7
        const int q = warp & 3, g = warp >> 2, r = 32 * q + lane;  // TMEM lane quadrant, group, row
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        bool ok = !aborted(abort_flag);
        float sx[16], sz = 0.f;
        if (ok && (ok = wait_w(abort_flag, &sm.qk_full))) {
            phi_tile_rolled<D>(sm.q, tid, kWork, len);
            phi_tile_rolled<D>(sm.k, tid, kWork, len);
            if (prm.dk < D) zero_cols<D>(sm.k, tid, kWork, prm.dk);
        }
        griddep_wait();
        griddep_launch_dependents();
        if (ok && (ok = wait_w(abort_flag, &sm.st_full))) {
            load_state(reinterpret_cast<const float *>(sm.dn), sm.zf, tid, sx, sz);
            put_state(sm.simg, sm.zf, sm.extra, tid, sx, sz);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kWork);  // zf[] complete before any thread of either group reads it
        if (ok) mbar_arrive(&sm.ready);
        // Both groups share every step: the conversions split by key blocks, the
        // epilogues by value columns [32 g, 32 g + 32) (named barrier 2 for the halves
        // of dO . o, 3 and 4 inside the conversions).
        const int c0 = 32 * g;
        if (ok) ok = wait_w(abort_flag, &sm.t_full);  // P = bf16(tril T)
        tc_fence_after();
        tmem_tril_bf16_split(ok, tl + tT, q, lane, g, 3, [](int) { return 0.f; });
        if (ok) {
            tc_fence_before();
            mbar_arrive(&sm.p_full);
        }
        float ddr = 0.f;
        if (ok && (ok = wait_w(abort_flag, &sm.full)) && (ok = wait_w(abort_flag, &sm.o_full))) {
            // o = num / d, dN = dO / d (bf16 into the dN tile), dd = -(dO . o) / d
            tc_fence_after();
            const float den = __uint_as_float(tmem_ld1(tl + tO + D)) + __uint_as_float(tmem_ld1(tl + tO + D + 1));
            tmem_ld_wait();
            const float inv = 1.f / fmaxf(den, prm.eps);
            float gsum = 0.f;
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                uint32_t a[16];
                tmem_ld16(tl + tO + c0 + 16 * blk, a);
                float go[16];
                ld_row16(sm.go, r, c0 + 16 * blk, go);
                tmem_ld_wait();
                float dnv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    gsum += go[e] * (__uint_as_float(a[e]) * inv);
                    dnv[e] = go[e] * inv;
                }
                st_row16(sm.dn, r, c0 + 16 * blk, dnv);
            }
            sm.gpart[g][r] = gsum;
        }
        named_bar_sync(2, kWork);
        if (ok) {
            const float den = __uint_as_float(tmem_ld1(tl + tO + D)) + __uint_as_float(tmem_ld1(tl + tO + D + 1));
            tmem_ld_wait();
            const float inv = 1.f / fmaxf(den, prm.eps);
            ddr = den > prm.eps ? -(sm.gpart[0][r] + sm.gpart[1][r]) * inv : 0.f;
            if (g == 0) {
                put_extra(sm.extra, r, kDdOff, pack_bf16(ddr, 0.f));
                if (r < len) ddbuf[(size_t)bh * prm.N + c * kC + r] = ddr;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.dn_ready);
        }
        if (ok && tid == 0 && (ok = wait_b(abort_flag, &sm.dn_ready))) {
            tma_store_3d_hint(&map_dn, sm.dn, 0, c * kC, bh, l2_policy_evict_last());
            tma_store_commit();
        }
        ok = __all_sync(0xffffffffu, ok);
        if (ok) ok = wait_w(abort_flag, &sm.u_full);  // U' = bf16(tril(U + dd 1^T))
        tc_fence_after();
        tmem_tril_bf16_split(ok, tl + tT, q, lane, g, 4, [ddr](int) { return ddr; });
        if (ok) {
            tc_fence_before();
            mbar_arrive(&sm.up_full);
        }
        if (ok && (ok = wait_w(abort_flag, &sm.bc_full)) && q < 2) {
            // B_c rows 0..63 (64..127 repeat them), value columns [c0, c0 + 32) and, for
            // group 0, the r column
            tc_fence_after();
            const int f = r;
            float4 *out = reinterpret_cast<float4 *>(slot);
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                uint32_t a[16];
                tmem_ld16(tl + tO + c0 + 16 * blk, a);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    out[((c0 + 16 * blk) / 4 + e) * D + f] = make_float4(
                        __uint_as_float(a[4 * e]), __uint_as_float(a[4 * e + 1]), __uint_as_float(a[4 * e + 2]),
                        __uint_as_float(a[4 * e + 3]));
            }
            if (g == 0) {
                slot[D * D + f] = __uint_as_float(tmem_ld1(tl + tO + D));
                tmem_ld_wait();
            }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (ok && (ok = wait_w(abort_flag, &sm.g_full))) {
            // dq = (dphi(Q) + dd z^T) phi'(q), staged in the dO tile (read only by the
            // output epilogue, long done)
            tc_fence_after();
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                uint32_t a[16];
                tmem_ld16(tl + tG + c0 + 16 * blk, a);
                float fq[16];
                ld_row16(sm.q, r, c0 + 16 * blk, fq);
                tmem_ld_wait();
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    x[e] = (__uint_as_float(a[e]) + ddr * sm.zf[c0 + 16 * blk + e]) * dphi(fq[e]);
                st_row16(sm.go, r, c0 + 16 * blk, x);
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.dq_staged);
        }
        if (tid == 0 && ok && wait_b(abort_flag, &sm.dq_staged)) {
            tma_store_3d_hint(&map_dq, sm.go, 0, c * kC, bh, l2_policy_evict_first());
            tma_store_commit();
        }
        if (tid == 0) tma_store_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------- 5. dk, dv
struct DkSmem {
    uint8_t q[kTile];   // phi(Q)
    uint8_t k[kTile];   // phi(K), then dk staged
    uint8_t v[kTile];
    uint8_t dn[kTile];  // dN, then dv staged
    uint8_t rimg[kImg]; // bf16 R after the chunk, [f][v]
    float rst[D * D];   // the fp32 R as copied
    float rf[D];        // r after the chunk (fp32)
    float dd[kC];
    // qk_full: Q, K landed; full: V, dN landed; st_full: the state landed
    uint64_t qk_full, full, st_full, ready, tt_full, ut_full, pt_full, upt_full, dv_full, dk_full, dv_staged, dk_staged, drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(DkSmem) + 1024 <= 232448 / 2, "two dk, dv CTAs per SM");

// TMEM of the dk, dv kernel: T^T at 0 (P^T over its first 64 columns, dV at 64),
// U^T at 128 (U'^T over its first 64 columns, dphi(K) at 192).
constexpr uint32_t tTT = 0, tDV = 64, tUT = 128, tDK = 192;

__global__ void __launch_bounds__(kThreads, 2)
bwd_tc_dkdv(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_dn,
            const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
            const float *buf, const float *ddbuf, const Params prm)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    DkSmem &sm = *reinterpret_cast<DkSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = (int)blockIdx.x / prm.nC, c = (int)blockIdx.x % prm.nC;
    const int len = min(kC, prm.N - c * kC);
    const float *slot = buf + ((size_t)bh * prm.nC + c) * kE;
    if (tid == 0) {
        uint64_t *bars[] = {&sm.qk_full, &sm.full, &sm.st_full, &sm.tt_full, &sm.ut_full, &sm.dv_full, &sm.dk_full, &sm.drain};
        for (uint64_t *b : bars) mbar_init(b, 1);
        mbar_init(&sm.ready, kWork);
        mbar_init(&sm.pt_full, 128);
        mbar_init(&sm.upt_full, 128);
        mbar_init(&sm.dv_staged, 128);
        mbar_init(&sm.dk_staged, 128);
        sm.abort = (smem_u32(smem_raw) & 1023u) == 0 ? 0 : 1;
        if (sm.abort) atomicOr(&g_bw_status, kStatusTimeout);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    int *abort_flag = &sm.abort;

    // As in the dq kernel: q, k, v, and dN and dd (the dq kernel's, which completed
    // before the scan preceding this grid passed its wait) are read before the wait;
    // the state R, which that scan writes, after it.
    if (warp == kTmaWarp) {
        const bool go = lane == 0 && !aborted(abort_flag);
        if (go) {
            const uint64_t pol = l2_policy_evict_first();
            mbar_arrive_expect_tx(&sm.qk_full, 2 * kTile);  // phi starts on these
            tma_load_3d_hint(sm.q, &map_q, &sm.qk_full, 0, c * kC, bh, pol);
            tma_load_3d_hint(sm.k, &map_k, &sm.qk_full, 0, c * kC, bh, pol);
            mbar_arrive_expect_tx(&sm.full, 2 * kTile);
            tma_load_3d_hint(sm.v, &map_v, &sm.full, 0, c * kC, bh, pol);
            tma_load_3d_hint(sm.dn, &map_dn, &sm.full, 0, c * kC, bh, pol);
        }
        griddep_wait();
        griddep_launch_dependents();
        if (go) {
            mbar_arrive_expect_tx(&sm.st_full, (D * D + D) * sizeof(float));
            bulk_load(sm.rst, slot, D * D * sizeof(float), &sm.st_full);
            bulk_load(sm.rf, slot + D * D, D * sizeof(float), &sm.st_full);
            drain(&sm.qk_full);
            drain(&sm.full);
            drain(&sm.st_full);
        }
    } else if (warp == kMmaWarp) {
        griddep_wait();
        griddep_launch_dependents();
        if (lane == 0) {
            const uint32_t qa = smem_u32(sm.q), ka = smem_u32(sm.k), va = smem_u32(sm.v), dna = smem_u32(sm.dn);
            const uint32_t ra = smem_u32(sm.rimg);
            bool ok = wait_b(abort_flag, &sm.ready);
            if (ok) {
                tc_fence_after();
                const uint32_t id = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + tTT, kmajor(ka, kk), kmajor(qa, kk), id, kk > 0);
                mma_commit(&sm.tt_full);  // T^T = phi(K) phi(Q)^T
                ok = wait_b(abort_flag, &sm.full);  // V, dN
            }
            if (ok) {
                tc_fence_after();
                const uint32_t id = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + tUT, kmajor(va, kk), kmajor(dna, kk), id, kk > 0);
                mma_commit(&sm.ut_full);  // U^T = V dN^T
            }
            if (ok && (ok = wait_b(abort_flag, &sm.pt_full))) {  // dV = P^T dN + phi(K) R
                tc_fence_after();
                const uint32_t id1 = idesc_bf16_f32(128, D, false, true);
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) mma_ts(tmem + tDV, tmem + tTT + kk * 8, mnmajor(dna, kk, 0), id1, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + tDV, kmajor(ka, kk), mnmajor(ra, kk, 0), id1, 1u);
                mma_commit(&sm.dv_full);
            }
            if (ok && (ok = wait_b(abort_flag, &sm.upt_full))) {  // dphi(K) = U'^T phi(Q) + V R^T
                tc_fence_after();
                const uint32_t id1 = idesc_bf16_f32(128, D, false, true);
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) mma_ts(tmem + tDK, tmem + tUT + kk * 8, mnmajor(qa, kk, 0), id1, kk > 0);
                const uint32_t id2 = idesc_bf16_f32(128, D, false, false);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + tDK, kmajor(va, kk), kmajor(ra, kk), id2, 1u);
                mma_commit(&sm.dk_full);
            }
            mma_commit(&sm.drain);
            drain(&sm.drain);
        }
    } else {
        // ---------------------------------------------------------------- warps 0-7
        const int q = warp & 3, g = warp >> 2, r = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        bool ok = !aborted(abort_flag);
        float sx[16], sz = 0.f, ddv = 0.f;
        if (ok && tid < kC && tid < len) ddv = __ldcg(ddbuf + (size_t)bh * prm.N + c * kC + tid);  // in flight during phi
        if (ok && (ok = wait_w(abort_flag, &sm.qk_full))) {
            phi_tile_rolled<D>(sm.q, tid, kWork, len);
            phi_tile_rolled<D>(sm.k, tid, kWork, len);
            if (prm.dk < D) zero_cols<D>(sm.k, tid, kWork, prm.dk);
        }
        griddep_wait();
        griddep_launch_dependents();
        if (ok && (ok = wait_w(abort_flag, &sm.st_full))) {
            load_state(sm.rst, sm.rf, tid, sx, sz);
            put_state(sm.rimg, sm.rf, nullptr, tid, sx, sz);
            if (tid < kC) sm.dd[tid] = ddv;
        }
        fence_proxy_async_smem();
        __syncwarp();
        named_bar_sync(1, kWork);  // dd[] complete before either group reads it
        if (ok) mbar_arrive(&sm.ready);
        if (g == 0) {
            // ---- group 0: P^T, dv
            if (ok && (ok = wait_w(abort_flag, &sm.tt_full))) {
                tc_fence_after();
                tmem_mask_bf16<false>(tl + tTT, q, lane, [](int) { return 0.f; });
                tc_fence_before();
                mbar_arrive(&sm.pt_full);
            }
            if (ok && (ok = wait_w(abort_flag, &sm.dv_full))) {
                tc_fence_after();
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    uint32_t a[16];
                    tmem_ld16(tl + tDV + 16 * blk, a);
                    tmem_ld_wait();
                    float x[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(a[e]);
                    st_row16(sm.dn, r, 16 * blk, x);  // dN is no longer read
                }
                fence_proxy_async_smem();
                mbar_arrive(&sm.dv_staged);
            }
            if (warp == 0 && lane == 0) {
                if (ok && wait_b(abort_flag, &sm.dv_staged)) {
                    tma_store_3d_hint(&map_dv, sm.dn, 0, c * kC, bh, l2_policy_evict_first());
                    tma_store_commit();
                }
                tma_store_wait_all();
            }
        } else {
            // ---- group 1: U'^T, dk
            if (ok && (ok = wait_w(abort_flag, &sm.ut_full))) {
                tc_fence_after();
                const float *ddp = sm.dd;
                tmem_mask_bf16<false>(tl + tUT, q, lane, [ddp](int col) { return ddp[col]; });
                tc_fence_before();
                mbar_arrive(&sm.upt_full);
            }
            if (ok && (ok = wait_w(abort_flag, &sm.dk_full))) {
                // dk = (dphi(K) + r^T) phi'(k), staged over phi(K) row by row (each thread reads
                // its row's phi values before overwriting them; every MMA has completed)
                tc_fence_after();
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    uint32_t a[16];
                    tmem_ld16(tl + tDK + 16 * blk, a);
                    float fk[16];
                    ld_row16(sm.k, r, 16 * blk, fk);
                    tmem_ld_wait();
                    float x[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = (__uint_as_float(a[e]) + sm.rf[16 * blk + e]) * dphi(fk[e]);
                    st_row16(sm.k, r, 16 * blk, x);
                }
                fence_proxy_async_smem();
                mbar_arrive(&sm.dk_staged);
            }
            if (warp == 4 && lane == 0) {
                if (ok && wait_b(abort_flag, &sm.dk_staged)) {
                    tma_store_3d_hint(&map_dk, sm.k, 0, c * kC, bh, l2_policy_evict_first());
                    tma_store_commit();
                }
                tma_store_wait_all();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// dk = dv = 64, or narrower widths (multiples of 8) on the same 64-column tiles: the
// zero-filled columns of q, k, v and dO enter phi(K) as 0 (zero_cols), so the forward
// quantities are exact; the terms phi(Q)'s extra columns feed (rows of R, columns of
// dphi(Q) and dphi(K)) land only in output columns past the widths, which the stores clip.
bool backward_tc_eligible(const BackwardProblem &p)
{
    return p.dtype == LA_BF16 && padded_widths_ok(p.dkd, p.dvd) && p.dkd <= D && p.dvd <= D && p.N >= kC;
}

la_status causal_backward_tc(const BackwardProblem &p)
{
    if (!backward_tc_eligible(p)) return LA_ERR_UNSUPPORTED;
    const int nC = ceil_div(p.N, kC);
    if ((long long)p.BH * nC > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    const size_t state_floats = (size_t)p.BH * nC * kE;
    const size_t dd_floats = (size_t)p.BH * p.N;
    const size_t dn_bytes = (size_t)p.BH * p.N * D * 2;
    // states, dd, then dN (16-byte aligned: the states and dd are multiples of 4 floats
    // only when N is; round the offset up).  The stream's data workspace when it can
    // serve the call (no allocation per call, none inside a captured graph), else
    // stream-ordered scratch.
    const size_t dn_off = ((sizeof(float) * (state_floats + dd_floats)) + 255) & ~(size_t)255;
    Scratch scratch;
    void *base = nullptr;
    la_status st = data_workspace(p.stream, dn_off + dn_bytes, &base);
    if (st != LA_OK) {
        st = scratch.alloc(dn_off + dn_bytes, p.stream);
        if (st != LA_OK) return st;
        base = scratch.ptr;
    }
    float *buf = (float *)base, *ddbuf = buf + state_floats;
    void *dn = (uint8_t *)base + dn_off;
    CUtensorMap mq, mk, mv, mdo, mdn, mdq, mdk, mdv;
    st = make_map(&mq, p.q, p.BH, p.N, p.dkd);
    if (st == LA_OK) st = make_map(&mk, p.k, p.BH, p.N, p.dkd);
    if (st == LA_OK) st = make_map(&mv, p.v, p.BH, p.N, p.dvd);
    if (st == LA_OK) st = make_map(&mdo, p.dout, p.BH, p.N, p.dvd);
    if (st == LA_OK) st = make_map(&mdn, dn, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mdq, p.dq, p.BH, p.N, p.dkd);
    if (st == LA_OK) st = make_map(&mdk, p.dk, p.BH, p.N, p.dkd);
    if (st == LA_OK) st = make_map(&mdv, p.dv, p.BH, p.N, p.dvd);
    if (st != LA_OK) return st;
    if (st == LA_OK) st = ensure_smem((const void *)bwd_tc_state, (int)sizeof(StateSmem));
    if (st == LA_OK) st = ensure_smem((const void *)bwd_tc_dq, (int)sizeof(DqSmem));
    if (st == LA_OK) st = ensure_smem((const void *)bwd_tc_dkdv, (int)sizeof(DkSmem));
    if (st != LA_OK) return st;
    Params prm{p.N, p.BH, nC, p.eps, p.dkd};
    const unsigned grid = (unsigned)(p.BH * nC);
    const unsigned scan_grid = (unsigned)(((long long)p.BH * (kE / 4) + kScanThreads - 1) / kScanThreads);
    count_launches(5);
    st = launch_dependent(bwd_tc_state, grid, kStateThreads, (int)sizeof(StateSmem), p.stream, mk, mv, buf, prm);
    if (st == LA_OK) st = launch_dependent(bwd_tc_scan, scan_grid, kScanThreads, 0, p.stream, buf, nC, p.BH, 0);
    if (st == LA_OK)
        st = launch_dependent(bwd_tc_dq, grid, kThreads, (int)sizeof(DqSmem), p.stream, mq, mk, mv, mdo, mdn, mdq, buf,
                              ddbuf, prm);
    if (st == LA_OK) st = launch_dependent(bwd_tc_scan, scan_grid, kScanThreads, 0, p.stream, buf, nC, p.BH, 1);
    if (st == LA_OK)
        st = launch_dependent(bwd_tc_dkdv, grid, kThreads, (int)sizeof(DkSmem), p.stream, mq, mk, mv, mdn, mdk, mdv, buf,
                              ddbuf, prm);
    return st;
}

la_status tc_backward_read_status(cudaStream_t s, unsigned *bits)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_bw_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_bw_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // namespace la
