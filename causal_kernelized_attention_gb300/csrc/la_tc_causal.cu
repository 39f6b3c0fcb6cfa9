// Tensor-core (tcgen05 + TMA) chunked causal forward, bf16 in / fp32 accumulate,
// dk = dv = D in {64, 128}, chunk C = 128.
//
// The chunked form ("Linear Attention", aiwiki.thehackersbrain.dev, listing
// linear_attention_chunked: quadratic and masked inside a chunk, recurrent
// across chunks; denominator = phi(Q_c) z + row sums of the masked scores,
// clamped) computed by one fused kernel:
//
//  * Work item = (b,h, segment of L chunks), taken in ticket order (segment-
//    major), one item per CTA.
//  * Phase A (segments with a successor): the segment's aggregate state
//    A_g = sum_c phi(K_c)^T V_c and a_g = sum_c colsum phi(K_c) accumulate in
//    tensor memory (TMEM).
//  * Phase B: wait (bounded) for the inclusive prefix P_{g-1} of the previous
//    segment of the same head, publish P_g = P_{g-1} + A_g, and load P_{g-1}
//    as the running state.  This is the exclusive scan of the chunk states,
//    done across segments, in fp32.
//  * Phase C: sweep the segment's chunks.  Per chunk c, on the tensor cores:
//      T   = phi(Q_c) phi(K_c)^T                         (fp32, TMEM)
//      P   = bf16(tril(T))                               (TMEM, written by threads)
//      O   = P V_c + phi(Q_c) bf16(S)                    (fp32, TMEM)
//      rs  = P 1,  qz = phi(Q_c) (z_hi + z_lo)           (denominator terms)
//      S  += phi(K_c)^T V_c,  z += phi(K_c)^T 1          (running state, fp32 TMEM)
//    o = O / max(rs + qz, eps), written as bf16.
//
// Warp roles (640 threads): warps 0-7 apply phi in shared memory; warp 8 issues
// TMA loads; warp 9 issues MMAs and owns TMEM; warps 12-15 turn T into P; warps
// 16-19 normalise O, refresh the bf16 copy of S and run phase B.  Waiting
// threads sleep on the mbarrier (suspend-time hint) rather than spin, so they
// leave issue slots to the working warps.  Every wait is bounded by
// %globaltimer; on expiry the CTA records LA_ERR_TIMEOUT in its status word,
// abandons its work, drains its in-flight copies and MMAs, and frees its TMEM.
#include "la_common.cuh"
#include "la_internal.h"
#include "la_sm100.cuh"

#include <algorithm>
#include <mutex>
#include <unordered_map>

namespace la {
namespace {

using namespace sm100;

static __device__ unsigned g_tc_status;

constexpr int kC = 128;                  // chunk (tokens per tile)
constexpr int kThreads = 640;
constexpr int kPhiThreads = 256;         // warps 0-7
constexpr int kTmaWarp = 8, kMmaWarp = 9, kEpiPWarp0 = 12, kEpiOWarp0 = 16;
constexpr uint32_t kSleepHintNs = 200000;  // per try_wait; the total wait stays bounded below
constexpr uint32_t kBox = kC * 128;      // one [128 rows x 64 bf16] swizzled box: 16 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any healthy wait
constexpr uint32_t kFlagReady = 1, kFlagError = 2;

template <int D>
struct Cfg {
    static constexpr int kStages = D == 128 ? 2 : 4;
    static constexpr uint32_t kTileBytes = kC * D * 2;
    static constexpr uint32_t kSbBytes = D * D * 2;   // bf16 copy of S, MN-major for the phi(Q) S MMA
    // TMEM columns
    static constexpr uint32_t tT = 0, tP = 128, tRS = 192, tQZ = 208, tZ = 224, tO = 256, tS = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
};

// W: [16 rows x 128] bf16, K-major, two 1 KB blocks of 8 rows (rows 8..15 of the
// descriptor alias into the next 2 KB, which is the S copy: only columns 0..2 of
// results that use W are read).  Row 0 = ones (row and column sums), rows 1 and 2 =
// the high and low bf16 parts of the running z.
template <int D>
struct alignas(1024) Smem {
    uint8_t q[Cfg<D>::kStages][Cfg<D>::kTileBytes];
    uint8_t k[Cfg<D>::kStages][Cfg<D>::kTileBytes];
    uint8_t v[Cfg<D>::kStages][Cfg<D>::kTileBytes];
    uint8_t w[2048];
    uint8_t sb[Cfg<D>::kSbBytes];
    uint64_t full[Cfg<D>::kStages], phi_done[Cfg<D>::kStages], empty[Cfg<D>::kStages];
    uint64_t t_full, t_free, p_full, o_full, o_free, s_full, s_ready, agg_ready, drain;
    uint32_t tmem_base;
    int ticket;
    int abort;
};

static_assert(sizeof(Smem<128>) <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
static_assert(sizeof(Smem<64>) <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

struct Params {
    uint16_t *o;            // bf16 output [BH, N, D]
    float *states;          // [BH, G, D*D + D] inclusive prefixes (S then z)
    uint32_t *flags;        // [BH, G]
    uint32_t *counter;      // work ticket
    int N, BH, G, L, n_chunks;
    float eps;
};

__device__ __forceinline__ bool aborted(const volatile int *a) { return *a != 0; }

// Bounded wait on an mbarrier phase; sets the CTA abort flag and the device
// status word on expiry.
__device__ __forceinline__ bool wait_bar(int *abort_flag, uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (aborted(abort_flag)) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *(volatile int *)abort_flag = 1;
            atomicOr(&g_tc_status, kStatusTimeout);
            return false;
        }
    }
}

// Same, with one result for the whole warp (for roles that issue warp-collective
// tcgen05.ld / tcgen05.st after the wait).
__device__ __forceinline__ bool wait_bar_warp(int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, wait_bar(abort_flag, bar, parity));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// phi on a pair of bf16 values: exp(min(x, 0)) + max(x, 0), which is x + 1 for
// x > 0 and exp(x) otherwise; min, max and the final add in packed bf16 (exact
// except the single rounding of the sum), exp in fp32.
__device__ __forceinline__ uint32_t phi2(uint32_t w)
{
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&w);
    const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
    const float2 nf = __bfloat1622float2(__hmin2(x, zero));
    const __nv_bfloat162 e = __floats2bfloat162_rn(__expf(nf.x), __expf(nf.y));
    const __nv_bfloat162 r = __hadd2(e, __hmax2(x, zero));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// phi in place on shared-memory tiles, by the 256 phi threads.  A unit is half of
// one 128-byte row of a 64-column box (4 chunks of 16 bytes); thread t takes units
// t, t + 256, ...  Units of rows >= `valid` (past the end of the sequence) are
// zeroed.  All loads of a thread are issued before its arithmetic.  The chunk
// order is rotated by the row so that the 8 threads of a quarter-warp (8
// consecutive rows) touch 8 different bank groups.
template <int D, int NU>
__device__ __forceinline__ void phi_tiles(uint8_t *kt, uint8_t *qt, int t, int valid)
{
    constexpr int kUnitsPerTile = 128 * (D / 32);
    uint4 buf[NU][4];
    uint8_t *rowp[NU];
    int rot[NU];
    bool ok[NU];
#pragma unroll
    for (int m = 0; m < NU; ++m) {
        const int u = t + kPhiThreads * m;
        uint8_t *tile = u < kUnitsPerTile ? kt : qt;
        const int rem = u % kUnitsPerTile, row = rem & 127, hb = rem >> 7;
        rowp[m] = tile + (hb >> 1) * kBox + row * 128;
        rot[m] = row + (hb & 1) * 4;
        ok[m] = row < valid;
#pragma unroll
        for (int k = 0; k < 4; ++k) buf[m][k] = *reinterpret_cast<const uint4 *>(rowp[m] + ((rot[m] + k) & 7) * 16);
    }
#pragma unroll
    for (int m = 0; m < NU; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 &x = buf[m][k];
            x = ok[m] ? make_uint4(phi2(x.x), phi2(x.y), phi2(x.z), phi2(x.w)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
    for (int m = 0; m < NU; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4 *>(rowp[m] + ((rot[m] + k) & 7) * 16) = buf[m][k];
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

template <int D>
__global__ void __launch_bounds__(640, 1)
causal_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 const __grid_constant__ CUtensorMap map_v, const Params prm)
{
    using CF = Cfg<D>;
    constexpr int S = CF::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // layout assumption of the swizzled tiles
        if (threadIdx.x == 0) atomicOr(&g_tc_status, kStatusTimeout);
        return;
    }
    Smem<D> &sm = *reinterpret_cast<Smem<D> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid < 128) {  // W: row 0 ones, everything else zero (rows 1, 2 get z in phase B)
        const int blk = tid >> 6, within = tid & 63;
        const uint32_t val = (within < 8) ? 0x3F803F80u : 0u;  // first 128 bytes of a block = row 0
        *reinterpret_cast<uint4 *>(sm.w + blk * 1024 + within * 16) = make_uint4(val, val, val, val);
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.phi_done[s], kPhiThreads);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.t_full, 1);
        mbar_init(&sm.t_free, 128);
        mbar_init(&sm.p_full, 128);
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.o_free, 128);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_ready, 128);
        mbar_init(&sm.agg_ready, 1);
        mbar_init(&sm.drain, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, CF::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The ticket is taken only once this CTA holds its TMEM, so a CTA that waits
    // on an earlier ticket waits on a CTA that is already running.
    if (tid == 0) sm.ticket = (int)atomicAdd(prm.counter, 1u);
    __syncthreads();

    const int ticket = sm.ticket;
    const int g = ticket / prm.BH, bh = ticket % prm.BH;
    const int c0 = g * prm.L;
    const int nch = min(prm.L, prm.n_chunks - c0);
    const bool has_next = g < prm.G - 1;  // phase A and publishing only when a successor exists
    const int nA = has_next ? nch : 0;
    const int total = nA + nch;
    const uint32_t tmem = sm.tmem_base;
    int *abort_flag = &sm.abort;

    if (warp < kPhiThreads / 32) {
        // ---------------------------------------------------------------- phi warps
        for (int j = 0; j < total; ++j) {
            const int s = j % S, r = j / S;
            if (!wait_bar(abort_flag, &sm.full[s], r & 1)) break;
            const bool isC = j >= nA;
            const int chunk = c0 + (isC ? j - nA : j);
            const int valid = prm.N - chunk * kC;
            if (isC)
                phi_tiles<D, D / 32>(sm.k[s], sm.q[s], tid, valid);
            else
                phi_tiles<D, D / 64>(sm.k[s], sm.q[s], tid, valid);
            fence_proxy_async_smem();
            mbar_arrive(&sm.phi_done[s]);
        }
    } else if (warp == kTmaWarp) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_map(&map_q);
            tma_prefetch_map(&map_k);
            tma_prefetch_map(&map_v);
            int issued = 0;
            for (int j = 0; j < total; ++j) {
                const int s = j % S, r = j / S;
                if (r > 0 && !wait_bar(abort_flag, &sm.empty[s], (r - 1) & 1)) break;
                const bool isC = j >= nA;
                const int row0 = (c0 + (isC ? j - nA : j)) * kC;
                mbar_arrive_expect_tx(&sm.full[s], (isC ? 3u : 2u) * CF::kTileBytes);
#pragma unroll
                for (int b = 0; b < D / 64; ++b) {
                    if (isC) tma_load_3d(sm.q[s] + b * kBox, &map_q, &sm.full[s], 64 * b, row0, bh);
                    tma_load_3d(sm.k[s] + b * kBox, &map_k, &sm.full[s], 64 * b, row0, bh);
                    tma_load_3d(sm.v[s] + b * kBox, &map_v, &sm.full[s], 64 * b, row0, bh);
                }
                issued = j + 1;
            }
            // No copy may still be writing shared memory when the CTA exits.
            for (int j = max(0, issued - S); j < issued; ++j) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&sm.full[j % S], (j / S) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_T = idesc_bf16_f32(128, 128, false, false);   // phi(Q) phi(K)^T
            const uint32_t id_PV = idesc_bf16_f32(128, D, false, true);     // P V (P in TMEM)
            const uint32_t id_QS = idesc_bf16_f32(128, D, false, true);     // phi(Q) S_bf16
            const uint32_t id_KV = idesc_bf16_f32(128, D, true, true);      // phi(K)^T V
            const uint32_t id_W = idesc_bf16_f32(128, 16, false, false);    // x W^T (A K-major or TMEM)
            const uint32_t id_KW = idesc_bf16_f32(128, 16, true, false);    // phi(K)^T W^T
            const uint32_t lbo_kt = kBox;  // second dk block of phi(K)^T (D = 64: rows 64..127 unused)
            const uint32_t w_addr = smem_u32(sm.w), sb_addr = smem_u32(sm.sb);
            bool ok = true;
            // phase A: aggregate state of the segment
            for (int ja = 0; ja < nA && ok; ++ja) {
                const int s = ja % S, r = ja / S;
                if (!(ok = wait_bar(abort_flag, &sm.phi_done[s], r & 1))) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(sm.k[s]), va = smem_u32(sm.v[s]);
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    const uint32_t acc = (ja > 0 || kk > 0) ? 1u : 0u;
                    mma_ss(tmem + CF::tS, mnmajor(ka, kk, lbo_kt), mnmajor(va, kk, kBox), id_KV, acc);
                    mma_ss(tmem + CF::tZ, mnmajor(ka, kk, lbo_kt), wdesc(w_addr, kk), id_KW, acc);
                }
                mma_commit(&sm.empty[s]);
            }
            if (ok && nA > 0) mma_commit(&sm.agg_ready);
            // phase C: outputs
            for (int cj = 0; cj < nch && ok; ++cj) {
                const int j = nA + cj, s = j % S, r = j / S;
                if (!(ok = wait_bar(abort_flag, &sm.phi_done[s], r & 1))) break;
                tc_fence_after();
                if (cj > 0 && !(ok = wait_bar(abort_flag, &sm.t_free, (cj - 1) & 1))) break;
                tc_fence_after();
                const uint32_t qa = smem_u32(sm.q[s]), ka = smem_u32(sm.k[s]), va = smem_u32(sm.v[s]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + CF::tT, kmajor(qa, kk), kmajor(ka, kk), id_T, kk > 0 ? 1u : 0u);
                mma_commit(&sm.t_full);
                if (cj > 0 && !(ok = wait_bar(abort_flag, &sm.o_free, (cj - 1) & 1))) break;
                if (!(ok = wait_bar(abort_flag, &sm.s_ready, cj & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    mma_ss(tmem + CF::tO, kmajor(qa, kk), mnmajor(sb_addr, kk, D * 128), id_QS, kk > 0 ? 1u : 0u);
                    mma_ss(tmem + CF::tQZ, kmajor(qa, kk), wdesc(w_addr, kk), id_W, kk > 0 ? 1u : 0u);
                }
                if (!(ok = wait_bar(abort_flag, &sm.p_full, cj & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    mma_ts(tmem + CF::tO, tmem + CF::tP + kk * 8, mnmajor(va, kk, kBox), id_PV, 1u);
                    mma_ts(tmem + CF::tRS, tmem + CF::tP + kk * 8, wdesc(w_addr, kk), id_W, kk > 0 ? 1u : 0u);
                }
                mma_commit(&sm.o_full);
                if (cj < nch - 1) {
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk) {
                        mma_ss(tmem + CF::tS, mnmajor(ka, kk, lbo_kt), mnmajor(va, kk, kBox), id_KV, 1u);
                        mma_ss(tmem + CF::tZ, mnmajor(ka, kk, lbo_kt), wdesc(w_addr, kk), id_KW, 1u);
                    }
                    mma_commit(&sm.s_full);
                }
                mma_commit(&sm.empty[s]);
            }
            // all issued MMAs complete before TMEM is freed
            mma_commit(&sm.drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&sm.drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else if (warp >= kEpiPWarp0 && warp < kEpiPWarp0 + 4) {
        // ---------------------------------------------------------------- T -> P
        const int quad = warp - kEpiPWarp0, i = quad * 32 + lane;  // query row = TMEM lane
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        for (int cj = 0; cj < nch; ++cj) {
            if (!wait_bar_warp(abort_flag, &sm.t_full, cj & 1)) break;
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t t[64];
                tmem_ld32(tl + CF::tT + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&t[0]));
                tmem_ld32(tl + CF::tT + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&t[32]));
                tmem_ld_wait();
                if (half == 1) {
                    tc_fence_before();
                    mbar_arrive(&sm.t_free);
                }
                uint32_t p[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int jk = half * 64 + 2 * e;  // key index within the chunk
                    const float a = jk <= i ? __uint_as_float(t[2 * e]) : 0.f;
                    const float b = jk + 1 <= i ? __uint_as_float(t[2 * e + 1]) : 0.f;
                    p[e] = pack_bf16(a, b);
                }
                tmem_st16(tl + CF::tP + half * 32, *reinterpret_cast<uint32_t(*)[16]>(&p[0]));
                tmem_st16(tl + CF::tP + half * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&p[16]));
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_full);
        }
    } else if (warp >= kEpiOWarp0) {
        // ---------------------------------------------------------------- phase B, O, S refresh
        const int quad = warp - kEpiOWarp0, i = quad * 32 + lane;  // query row / state row = TMEM lane
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        const size_t seg_floats = (size_t)D * D + D;
        const bool row_ok = i < D;

        // Writes row i of the bf16 state copy (32 columns starting at c0) and the z split.
        auto put_sb = [&](int col0, const float *x) {
#pragma unroll
            for (int c8 = 0; c8 < 32; c8 += 8) {
                const int col = col0 + c8;
                const uint32_t off = (col >> 6) * (D * 128) + i * 128 + ((((col & 63) >> 3) ^ (i & 7)) << 4);
                *reinterpret_cast<uint4 *>(sm.sb + off) =
                    make_uint4(pack_bf16(x[c8], x[c8 + 1]), pack_bf16(x[c8 + 2], x[c8 + 3]),
                               pack_bf16(x[c8 + 4], x[c8 + 5]), pack_bf16(x[c8 + 6], x[c8 + 7]));
            }
        };
        auto put_z = [&](float zv) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
            const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
            uint8_t *blk = sm.w + (i >> 6) * 1024;
            *reinterpret_cast<__nv_bfloat16 *>(blk + sw128_offset(1, i & 63)) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(blk + sw128_offset(2, i & 63)) = lo;
        };

        // ---- phase B: prefix of the earlier segments of this head
        const float *prev = nullptr;
        bool failed = false;
        if (g > 0) {
            if (i == 0) {
                const uint32_t *f = prm.flags + (size_t)bh * prm.G + (g - 1);
                const uint64_t t0 = globaltimer_ns();
                uint32_t v = ld_acquire_gpu(f);
                while (v == 0) {
                    if (globaltimer_ns() - t0 > kWaitLimitNs) {
                        atomicOr(&g_tc_status, kStatusTimeout);
                        v = kFlagError;
                        break;
                    }
                    __nanosleep(256);
                    v = ld_acquire_gpu(f);
                }
                if (v != kFlagReady) *(volatile int *)abort_flag = 1;
            }
            named_bar_sync(1, 128);
            failed = aborted(abort_flag);
            if (!failed) prev = prm.states + ((size_t)bh * prm.G + (g - 1)) * seg_floats;
        }
        float *mine = has_next ? prm.states + ((size_t)bh * prm.G + g) * seg_floats : nullptr;
        bool have_agg = false;
        if (nA > 0) have_agg = wait_bar_warp(abort_flag, &sm.agg_ready, 0);
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
            float pv[32];
            if (prev != nullptr && row_ok) {
                const float4 *src = reinterpret_cast<const float4 *>(prev + (size_t)i * D + cc * 32);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 x = __ldcg(src + e);
                    pv[4 * e] = x.x; pv[4 * e + 1] = x.y; pv[4 * e + 2] = x.z; pv[4 * e + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) pv[e] = 0.f;
            }
            if (have_agg) {
                uint32_t a[32];
                tmem_ld32(tl + CF::tS + cc * 32, a);
                tmem_ld_wait();
                if (row_ok) {
                    float4 *dst = reinterpret_cast<float4 *>(mine + (size_t)i * D + cc * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(pv[4 * e] + __uint_as_float(a[4 * e]),
                                             pv[4 * e + 1] + __uint_as_float(a[4 * e + 1]),
                                             pv[4 * e + 2] + __uint_as_float(a[4 * e + 2]),
                                             pv[4 * e + 3] + __uint_as_float(a[4 * e + 3]));
                }
            }
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                w0[e] = __float_as_uint(pv[e]);
                w1[e] = __float_as_uint(pv[16 + e]);
            }
            tmem_st16(tl + CF::tS + cc * 32, w0);
            tmem_st16(tl + CF::tS + cc * 32 + 16, w1);
            if (row_ok) put_sb(cc * 32, pv);
        }
        {
            const float zp = (prev != nullptr && row_ok) ? __ldcg(prev + (size_t)D * D + i) : 0.f;
            if (have_agg) {
                const float za = __uint_as_float(tmem_ld1(tl + CF::tZ));
                tmem_ld_wait();
                if (row_ok) mine[(size_t)D * D + i] = zp + za;
            }
            tmem_st1(tl + CF::tZ, __float_as_uint(zp));
            if (row_ok) put_z(zp);
        }
        tmem_st_wait();
        if (has_next) {
            __threadfence();
            named_bar_sync(1, 128);
            if (i == 0)
                st_release_gpu(prm.flags + (size_t)bh * prm.G + g,
                               (have_agg && !aborted(abort_flag)) ? kFlagReady : kFlagError);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.s_ready);

        // ---- phase C: normalise and store O; refresh the bf16 state copy
        for (int cj = 0; cj < nch; ++cj) {
            if (!wait_bar_warp(abort_flag, &sm.o_full, cj & 1)) break;
            tc_fence_after();
            uint32_t dn[32];
            tmem_ld32(tl + CF::tRS, dn);  // columns: rs[0..15], qz[0..15]
            tmem_ld_wait();
            const float den = __uint_as_float(dn[0]) + __uint_as_float(dn[17]) + __uint_as_float(dn[18]);
            const float inv = 1.f / fmaxf(den, prm.eps);
            const int row = (c0 + cj) * kC + i;
            uint16_t *orow = prm.o + ((size_t)bh * prm.N + row) * D;
#pragma unroll 1
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t a[64];
                tmem_ld32(tl + CF::tO + cc * 64, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
                tmem_ld32(tl + CF::tO + cc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&a[32]));
                tmem_ld_wait();
                if (row < prm.N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 64);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_uint4(
                            pack_bf16(__uint_as_float(a[8 * e]) * inv, __uint_as_float(a[8 * e + 1]) * inv),
                            pack_bf16(__uint_as_float(a[8 * e + 2]) * inv, __uint_as_float(a[8 * e + 3]) * inv),
                            pack_bf16(__uint_as_float(a[8 * e + 4]) * inv, __uint_as_float(a[8 * e + 5]) * inv),
                            pack_bf16(__uint_as_float(a[8 * e + 6]) * inv, __uint_as_float(a[8 * e + 7]) * inv));
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.o_free);
            if (cj < nch - 1) {
                if (!wait_bar_warp(abort_flag, &sm.s_full, cj & 1)) break;
                tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < D / 64; ++cc) {
                    uint32_t a[64];
                    tmem_ld32(tl + CF::tS + cc * 64, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
                    tmem_ld32(tl + CF::tS + cc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&a[32]));
                    tmem_ld_wait();
                    if (row_ok) {
                        put_sb(cc * 64, reinterpret_cast<const float *>(&a[0]));
                        put_sb(cc * 64 + 32, reinterpret_cast<const float *>(&a[32]));
                    }
                }
                const float zv = __uint_as_float(tmem_ld1(tl + CF::tZ));
                tmem_ld_wait();
                if (row_ok) put_z(zv);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&sm.s_ready);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, CF::kTmemCols);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

la_status encode_fn(EncodeTiledFn *out)
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

// [BH, N, D] bf16 as a 3-D tensor (D, N, BH); box = 64 columns x 128 rows, 128-byte swizzle.
la_status make_map(CUtensorMap *m, const void *ptr, int BH, int N, int D)
{
    EncodeTiledFn enc;
    la_status st = encode_fn(&enc);
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

int sm_count()
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

template <int D>
la_status launch(const Problem &p)
{
    CUtensorMap mq, mk, mv;
    la_status st = make_map(&mq, p.q, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mk, p.k, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mv, p.v, p.BH, p.N, D);
    if (st != LA_OK) return st;

    const int n_chunks = ceil_div(p.N, kC);
    const long long work = (long long)p.BH * n_chunks;
    const int L = (int)std::min<long long>(8, std::max<long long>(1, (work + sm_count() - 1) / sm_count()));
    const int G = ceil_div(n_chunks, L);
    const size_t items = (size_t)p.BH * G;
    const size_t flag_bytes = ((items * 4 + 16) + 255) / 256 * 256;
    const size_t state_bytes = G > 1 ? items * ((size_t)D * D + D) * 4 : 0;

    Scratch scratch;
    st = scratch.alloc(flag_bytes + state_bytes, p.stream);
    if (st != LA_OK) return st;
    uint8_t *base = (uint8_t *)scratch.ptr;
    cudaError_t e = cudaMemsetAsync(base, 0, flag_bytes, p.stream);
    count_launches();
    if (e != cudaSuccess) return cuda_status(e);

    Params prm;
    prm.o = (uint16_t *)p.o;
    prm.counter = (uint32_t *)base;
    prm.flags = (uint32_t *)(base + 16);
    prm.states = (float *)(base + flag_bytes);
    prm.N = p.N;
    prm.BH = p.BH;
    prm.G = G;
    prm.L = L;
    prm.n_chunks = n_chunks;
    prm.eps = p.eps;

    const int smem = (int)sizeof(Smem<D>);
    auto kern = causal_tc_kernel<D>;
    st = ensure_smem((const void *)kern, smem);
    if (st != LA_OK) return st;
    count_launches();
    kern<<<(unsigned)items, kThreads, smem, p.stream>>>(mq, mk, mv, prm);
    return cuda_status(cudaGetLastError());
}

}  // namespace

la_status causal_tc(const Problem &p)
{
    if (p.dtype != LA_BF16 || p.dk != p.dv || (p.dk != 64 && p.dk != 128) || p.chunk != kC || p.N < kC)
        return LA_ERR_UNSUPPORTED;
    return p.dk == 128 ? launch<128>(p) : launch<64>(p);
}

la_status tc_causal_read_status(cudaStream_t s, unsigned *bits)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_tc_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // namespace la
