// Tensor-core causal forward for sequences of up to 16 chunks (bf16 in / fp32
// accumulate, dk = dv = 64, chunk C = 128, 128 <= N <= 2048): one thread-block
// cluster of 4 CTAs per head, the exclusive scan of the chunk states exchanged
// through distributed shared memory.
//
// The chunked form ("Linear Attention", aiwiki.thehackersbrain.dev, listing
// linear_attention_chunked; "Linear Attention -- Math + Variants", Chunkwise
// parallelism): the masked quadratic form inside a chunk, the state
// S = sum phi(k) v^T, z = sum phi(k) across chunks.
//
//  * CTA r of a head's cluster holds the head's chunks [r L, (r+1) L),
//    L = ceil(n_c / 4) <= 4, all of them in shared memory at once (Q, K and V
//    loaded by TMA at the start; O is later staged in each chunk's Q tile).
//  * Phase A, on the tensor cores: the state of chunk p, phi(K_p)^T [V_p | 1], in
//    its own TMEM columns (its rows repeated in the upper lanes, so that every lane
//    quadrant sees all 64 key features); the scan threads read the four back once
//    and form the running sums after each chunk in registers.
//  * Scan: each CTA puts its segment total (fp32) in its shared memory, and the
//    CTAs of higher rank add up the totals of the lower ranks straight from their
//    shared memory (ld.shared::cluster), synchronised by remote mbarrier arrivals
//    with release / acquire at cluster scope: E_r, the state before the segment.
//  * Output, on the tensor cores, for chunk p of the segment with image
//    bf16(E_r + running sum up to chunk p - 1) (and z as a bf16 high + low pair):
//      T = phi(Q_p) phi(K_p)^T,  P = bf16(tril T) over T in TMEM,
//      O = P [V_p | 1] + phi(Q_p) [image | z],  o = O / max(rowsum + phi(q) z, eps).
//    Only phi(Q) [image | z] waits for the scan.  The images go into each chunk's
//    K tile once T of that chunk (and of its pair) has completed, two chunks at a
//    time, so no chunk waits on the chunk before it.
//
// Warp roles (512 threads): warps 0-3 and 4-7 are two groups that each cover the
// four TMEM lane quadrants.  Together (256 threads) they apply phi to every K tile
// as it lands, read the chunk states, do the scan and write the images; group g
// turns T into P and normalises and stores O for the chunks p with p % 2 == g.
// Warp 8: TMA.  Warp 9: MMA issue and TMEM.  Warps 10-12, 14, 15: phi of the Q
// tiles (warp 13, on the MMA warp's sub-partition, idles).  The order within the
// groups was set by a %globaltimer trace of the launch: phi of K first (the
// groups are otherwise idle while the loads land), the segment total published
// right after phase A, T -> P of the group's first chunk before the cross-CTA sum
// (the sum's distributed-shared-memory reads take about 0.6 us for the highest
// rank), and T -> P of the second chunk after the first images.  In the tail the
// MMA issue thread is the limit: each group of 4 or 8 MMAs takes 400-600 cycles
// from the first issue to the commit.
//
// Every wait is bounded (Params::wait_ns); on expiry the CTA records LA_ERR_TIMEOUT
// in this file's status word and winds down.  No CTA returns early: every one
// reaches the final cluster barrier, so none leaves while a peer may still read its
// shared memory or arrive on its barriers.
#include "la_common.cuh"
#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"

#include <algorithm>
#include <cstddef>

namespace la {
namespace {

using namespace sm100;
using namespace tc;

static __device__ unsigned g_cl_status;

constexpr int D = 64;
constexpr int kG = 4;                    // CTAs per cluster (one head)
constexpr int kLmax = 4;                 // chunks per CTA
constexpr int kThreads = 512;
constexpr uint32_t kTile = kC * D * 2;   // 16 KB
constexpr uint32_t kSbBytes = D * D * 2; // 8 KB bf16 image
constexpr int kTmaWarp = 8, kMmaWarp = 9, kPhiWarp0 = 10;
constexpr int kScanThreads = 256, kPhiThreads = 160;
// The phi warps are 10, 11, 12, 14 and 15: warp 13 would share a sub-partition (warp
// index mod 4) with the MMA warp, whose issue rate drops severalfold while another
// warp of its sub-partition has work; it stays idle.
constexpr int kIdleWarp = 13;
static_assert(kIdleWarp % 4 == kMmaWarp % 4, "the idle warp shares the MMA warp's sub-partition");

// TMEM columns.  T / P buffers at 0 and 128; O buffers at 256, 336 and 416 (chunk
// 2; chunk 3 reuses chunk 1's).  Phase A puts chunk p's state in its own group of 80
// columns, the first three in the T / P area and the fourth at 416; all are read
// before the first T is issued.  (Keeping the T / P buffers clear, so that T(0) need
// not wait for the read, measured 0.4 us slower per launch.)
constexpr uint32_t tO0 = 256, tO1 = 336, tA3 = 416;
__host__ __device__ constexpr uint32_t a_col(int p) { return p < 3 ? 80u * (uint32_t)p : tA3; }
// O buffer of chunk p (0: chunk 0, 1: chunks 1 and 3, 2: chunk 2) and its column
__host__ __device__ constexpr int o_buf(int p) { return p == 0 ? 0 : p == 2 ? 2 : 1; }
__host__ __device__ constexpr uint32_t o_col(int b) { return b == 0 ? tO0 : b == 1 ? tO1 : tA3; }
static_assert(a_col(2) + 80 <= tO0 && tO0 + 80 <= tO1 && tO1 + 80 <= tA3 && tA3 + 80 <= 512,
              "TMEM column groups overlap");
constexpr uint32_t kDrainNs = 100000000u;

struct alignas(1024) Smem {
    uint8_t q[kLmax][kTile];
    uint8_t k[kLmax][kTile];
    uint8_t v[kLmax][kTile];
    // this CTA's segment total for its peers: fp32 S in the thread-major layout
    // (the float4 of columns 4c..4c+3 of row i at float4 index c * D + i), and z
    float4 xch[D * D / 4];
    // column 0 = 1 (the row sums of P); a 128-byte-swizzled operand, so 1024-byte aligned
    alignas(1024) uint8_t ones[kC * 128];
    float xz[D];
    uint64_t kv_full[kLmax], q_full[kLmax], k_ready[kLmax], q_ready[kLmax];
    uint64_t a_full, a_read, drain;  // phase A done (one-shot); its states read (one-shot)
    uint64_t t_full[2], p_full[2], pv_done[2];
    uint64_t o_full[3], o_staged[3], o_free;  // per O buffer; o_free: buffer 1 read (chunk 1)
    uint64_t t_done[2];     // T of chunks 2 j, 2 j + 1 completed (one-shot, from the MMA warp)
    uint64_t img_ready[2];  // the images of chunks 2 j, 2 j + 1 are in place (one-shot)
    uint64_t scan_sync;  // the scan threads' barrier (bounded)
    uint64_t agg_ready;  // the lower ranks' totals are readable (their remote arrivals)
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Smem) <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
static_assert(offsetof(Smem, ones) % 1024 == 0 && offsetof(Smem, k) % 1024 == 0, "swizzled operands 1024-aligned");
// a chunk's image (8 KB) and its z block (8 KB) fill the chunk's K tile
static_assert(2 * kSbBytes == kTile, "image and z block fill a K tile");

struct Params {
    int N, BH, n_c, L;
    float eps;
    unsigned long long wait_ns;
    // Feature-map variant (kVar): LA_PHI_* map with the shift as a bf16 pair; normalize 0:
    // o = phi(q)^T S without the denominator.
    int map, normalize;
    uint32_t shift2;
};

// phi (elu + 1, or with kVar the map `map` with shift c2) in place on one tile, as a
// loop that is not unrolled (its code is fetched once per launch), by nt threads.
template <bool kVar>
__device__ __forceinline__ void phi_tile_cluster(uint8_t *tile, int t, int nt, int valid, const Params &prm)
{
    if (!kVar) {
        phi_tile_rolled<D>(tile, t, nt, valid);
        return;
    }
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
            x[k] = live ? make_uint4(phi2_variant(x[k].x, prm.map, prm.shift2), phi2_variant(x[k].y, prm.map, prm.shift2),
                                     phi2_variant(x[k].z, prm.map, prm.shift2), phi2_variant(x[k].w, prm.map, prm.shift2))
                        : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4 *>(rp + ((rot + k) & 7) * 16) = x[k];
    }
}

__device__ __forceinline__ bool wait_bar(const Params &prm, int *abort_flag, uint64_t *bar, uint32_t parity,
                                         bool cluster_acquire = false)
{
    auto done = [&]() { return cluster_acquire ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (done()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (cluster_acquire ? done() : mbar_try_wait_sleep(bar, parity, 20000)) return true;
        if (aborted(abort_flag)) return false;
        if (globaltimer_ns() - t0 > prm.wait_ns) {
            *(volatile int *)abort_flag = 1;
            atomicOr(&g_cl_status, kStatusTimeout);
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bar_warp(const Params &prm, int *abort_flag, uint64_t *bar, uint32_t parity,
                                              bool cluster_acquire = false)
{
    return __all_sync(0xffffffffu, wait_bar(prm, abort_flag, bar, parity, cluster_acquire));
}
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < kDrainNs) {
    }
}
// The scan threads' barrier: an mbarrier of 256 arrivals waited on with a bound.
__device__ __forceinline__ bool scan_barrier(const Params &prm, Smem &sm, int *abort_flag, uint32_t &uses)
{
    mbar_arrive(&sm.scan_sync);
    const bool ok = wait_bar_warp(prm, abort_flag, &sm.scan_sync, uses & 1);
    ++uses;
    return ok;
}

// Row i of a z block: the second 64-wide block of the [image | z] operand, of
// which the MMA reads columns 0..15 -- z_i as a bf16 high + low pair in columns 0
// and 1, zeros in 2..15 (128-byte swizzled rows, 16-byte chunks 0 and 1).
__device__ __forceinline__ void put_z_row(uint8_t *zb, int i, float zv)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
    const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
    const __nv_bfloat162 pair = __halves2bfloat162(hi, lo);
    uint8_t *row = zb + i * 128;
    *reinterpret_cast<uint4 *>(row + ((0 ^ (i & 7)) << 4)) =
        make_uint4(*reinterpret_cast<const uint32_t *>(&pair), 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(row + ((1 ^ (i & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
}
// Row i, columns [col0, col0 + 16) of a bf16 image (MN-major, 128-byte swizzled, D = 64).
__device__ __forceinline__ void put_img16(uint8_t *sb, int i, int col0, const float (&x)[16])
{
#pragma unroll
    for (int c8 = 0; c8 < 16; c8 += 8) {
        const int col = col0 + c8;
        *reinterpret_cast<uint4 *>(sb + i * 128 + (((col >> 3) ^ (i & 7)) << 4)) =
            make_uint4(pack_bf16(x[c8], x[c8 + 1]), pack_bf16(x[c8 + 2], x[c8 + 3]), pack_bf16(x[c8 + 4], x[c8 + 5]),
                       pack_bf16(x[c8 + 6], x[c8 + 7]));
    }
}


template <bool kVar>
__global__ void __launch_bounds__(kThreads, 1)
causal_cluster_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                      const Params prm)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // (no early return: every CTA must reach the cluster barriers)
    const bool layout_ok = (smem_u32(smem_raw) & 1023u) == 0;
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    const int bh = (int)blockIdx.x / kG;
    const int c0 = rank * prm.L;
    const int nch = max(0, min(prm.L, prm.n_c - c0));
    griddep_launch_dependents();

    if (tid < 128) {
        for (int c = tid; c < kC * 8; c += 128) {
            const uint32_t x = (c & 7) == ((c >> 3) & 7) ? 0x3F80u : 0u;
            *reinterpret_cast<uint4 *>(sm.ones + c * 16) = make_uint4(x, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        for (int p = 0; p < kLmax; ++p) {
            mbar_init(&sm.kv_full[p], 1);
            mbar_init(&sm.q_full[p], 1);
            mbar_init(&sm.k_ready[p], kScanThreads);
            mbar_init(&sm.q_ready[p], kPhiThreads);
        }
        mbar_init(&sm.a_full, 1);
        mbar_init(&sm.a_read, kScanThreads);
        mbar_init(&sm.o_free, 128);
        for (int b = 0; b < 3; ++b) {
            mbar_init(&sm.o_full[b], 1);
            mbar_init(&sm.o_staged[b], 128);
        }
        mbar_init(&sm.drain, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.t_full[b], 1);
            mbar_init(&sm.p_full[b], 128);
            mbar_init(&sm.pv_done[b], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&sm.t_done[j], 1);
            mbar_init(&sm.img_ready[j], kScanThreads);
        }
        mbar_init(&sm.scan_sync, kScanThreads);
        mbar_init(&sm.agg_ready, max(rank, 1));  // one arrival per lower rank
        sm.abort = layout_ok ? 0 : 1;
        if (!layout_ok) atomicOr(&g_cl_status, kStatusTimeout);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == kTmaWarp && lane == 0) {
        // the tensor maps are launch parameters and the L2 is coherent: both prefetches
        // may run while an earlier kernel on the stream still writes the inputs
        tma_prefetch_map(&map_q);
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
        tma_prefetch_map(&map_o);
        for (int p = 0; p < nch; ++p) {
            tma_prefetch_3d(&map_k, 0, (c0 + p) * kC, bh);
            tma_prefetch_3d(&map_v, 0, (c0 + p) * kC, bh);
        }
        for (int p = 0; p < nch; ++p) tma_prefetch_3d(&map_q, 0, (c0 + p) * kC, bh);
    }
    griddep_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // every CTA of the cluster has initialised its barriers before any peer arrives on them
    cluster_sync_all();
    const uint32_t tmem = sm.tmem_base;
    int *abort_flag = &sm.abort;

    if (warp == kIdleWarp) {
        // nothing: see kIdleWarp
    } else if (warp >= kPhiWarp0) {
        // ---------------------------------------------------------------- phi warps: every Q tile
        // (warps 0-7 take every K tile as it lands)
        const int t = (warp - kPhiWarp0 - (warp > kIdleWarp ? 1 : 0)) * 32 + lane;
        bool ok = true;
#pragma unroll 1
        for (int p = 0; p < nch && ok; ++p) {
            if (!(ok = wait_bar_warp(prm, abort_flag, &sm.q_full[p], 0))) break;
            phi_tile_cluster<kVar>(sm.q[p], t, kPhiThreads, prm.N - (c0 + p) * kC, prm);
            fence_proxy_async_smem();
            mbar_arrive(&sm.q_ready[p]);
        }
    } else if (warp == kTmaWarp) {
        // ---------------------------------------------------------------- TMA: the whole segment at once
        if (lane == 0 && !aborted(abort_flag)) {
            tma_prefetch_map(&map_q);
            tma_prefetch_map(&map_k);
            tma_prefetch_map(&map_v);
            tma_prefetch_map(&map_o);
            const uint64_t pol = l2_policy_evict_first();  // every tile is read once
            for (int p = 0; p < nch; ++p) {
                mbar_arrive_expect_tx(&sm.kv_full[p], 2 * kTile);
                tma_load_3d_hint(sm.k[p], &map_k, &sm.kv_full[p], 0, (c0 + p) * kC, bh, pol);
                tma_load_3d_hint(sm.v[p], &map_v, &sm.kv_full[p], 0, (c0 + p) * kC, bh, pol);
            }
            for (int p = 0; p < nch; ++p) {
                mbar_arrive_expect_tx(&sm.q_full[p], kTile);
                tma_load_3d_hint(sm.q[p], &map_q, &sm.q_full[p], 0, (c0 + p) * kC, bh, pol);
            }
            // no copy may still be writing shared memory when the CTA exits
            for (int p = 0; p < nch; ++p) {
                drain_bar(&sm.kv_full[p], 0);
                drain_bar(&sm.q_full[p], 0);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_T = idesc_bf16_f32(128, 128, false, false);    // phi(Q) phi(K)^T
            const uint32_t id_PV = idesc_bf16_f32(128, D + 16, false, true); // P [V | 1] (P in TMEM)
            const uint32_t id_QS = idesc_bf16_f32(128, D + 16, false, true); // phi(Q) [image | z]
            const uint32_t id_KV = idesc_bf16_f32(128, D + 16, true, true);  // phi(K)^T [V | 1]
            const uint32_t ones = smem_u32(sm.ones);
            bool ok = true;
            // Phase A: the state of each chunk in its own columns.  phi(K)^T is MN-major;
            // its second 64-row block has offset 0 (LBO = 0), so rows 64..127 of each
            // state repeat rows 0..63.
#pragma unroll 1
            for (int p = 0; p < nch && ok; ++p) {
                if (!(ok = wait_bar(prm, abort_flag, &sm.k_ready[p], 0))) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(sm.k[p]), va = smem_u32(sm.v[p]);
                const uint64_t dkt = mnmajor(ka, 0, 0), dv = mnmajor(va, 0, ones - va);
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_ss(tmem + a_col(p), dkt + 128 * kk, dv + 128 * kk, id_KV, kk > 0 ? 1u : 0u);
            }
            if (ok && nch > 0) mma_commit(&sm.a_full);
            auto issue_T = [&](int p) -> bool {
                if (!wait_bar(prm, abort_flag, &sm.q_ready[p], 0)) return false;
                if (p >= 2 && !wait_bar(prm, abort_flag, &sm.pv_done[p & 1], ((p - 2) >> 1) & 1)) return false;
                tc_fence_after();
                const uint64_t dq = kmajor(smem_u32(sm.q[p]), 0), dk = kmajor(smem_u32(sm.k[p]), 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + (p & 1) * 128, dq + 2 * kk, dk + 2 * kk, id_T, kk > 0 ? 1u : 0u);
                mma_commit(&sm.t_full[p & 1]);
                return true;
            };
            auto issue_PV = [&](int p) -> bool {
                if (!wait_bar(prm, abort_flag, &sm.p_full[p & 1], (p >> 1) & 1)) return false;
                if (p == 3 && !wait_bar(prm, abort_flag, &sm.o_free, 0)) return false;  // chunk 1's O read
                tc_fence_after();
                const uint32_t va = smem_u32(sm.v[p]);
                const uint64_t dv = mnmajor(va, 0, ones - va);
                const uint32_t dO = tmem + o_col(o_buf(p)), dP = tmem + (p & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) mma_ts(dO, dP + kk * 8, dv + 128 * kk, id_PV, kk > 0 ? 1u : 0u);
                if (p < 2) mma_commit(&sm.pv_done[p & 1]);  // only T(p + 2) waits for it
                return true;
            };
            auto issue_QS = [&](int p) -> bool {
                tc_fence_after();
                if (c0 + p > 0) {  // the head's first chunk has no state before it
                    // [image | z]: the image in the first half of the chunk's K tile, the
                    // z block in the second half (an LBO of 8 KB)
                    const uint64_t dsb = mnmajor(smem_u32(sm.k[p]), 0, kSbBytes);
                    const uint64_t dq = kmajor(smem_u32(sm.q[p]), 0);
                    const uint32_t dO = tmem + o_col(o_buf(p));
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) mma_ss(dO, dq + 2 * kk, dsb + 128 * kk, id_QS, 1u);
                }
                mma_commit(&sm.o_full[o_buf(p)]);
                return true;
            };
            // Before the scan: T of every chunk and P V of the first two (their O buffers
            // are free); T of chunk p >= 2 needs P V of chunk p - 2 done with its buffer.
            const int pre = min(2, nch);
            if (ok && nch > 0) ok = wait_bar(prm, abort_flag, &sm.a_read, 0);
            for (int p = 0; p < pre && ok; ++p) ok = issue_T(p);
            if (ok) mma_commit(&sm.t_done[0]);
            for (int p = 0; p < pre && ok; ++p) ok = issue_PV(p);
            for (int p = 2; p < nch && ok; ++p) ok = issue_T(p);
            if (ok) mma_commit(&sm.t_done[1]);
            // After the scan: the state term of each chunk once its pair's images are in
            // place (and P V of chunks 2, 3, whose O buffers free up as the first
            // outputs are written).
            for (int p = 0; p < nch && ok; ++p) {
                if (p >= 2 && !(ok = issue_PV(p))) break;
                if ((p & 1) == 0 && !(ok = wait_bar(prm, abort_flag, &sm.img_ready[p >> 1], 0))) break;
                ok = issue_QS(p);
            }
            // all issued MMAs complete before TMEM is freed
            mma_commit(&sm.drain);
            drain_bar(&sm.drain, 0);
        }
    } else {
        // ---------------------------------------------------------------- warps 0-7: scan, T->P, O
        // Scan mapping: thread s owns row i = 32 (q % 2) + lane of the states and
        // columns [16 h, 16 h + 16), with q = warp % 4 its TMEM lane quadrant and
        // h = 2 (warp / 4) + q / 2; h = 0 also owns z_i.
        const int q = warp & 3;
        const int i = 32 * (q & 1) + lane, h = 2 * (warp >> 2) + (q >> 1);
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        uint32_t syncs = 0;
        bool ok = true;
        // ---- phase A: the chunk states, read once all are in place; the running sums
        // after chunks 0 .. L-2 stay in registers for the images, the one after the
        // last chunk is the segment total, which goes to the exchange buffer.
        float cum[kLmax - 1][16], cz[kLmax - 1];
        float4 *xb = sm.xch;
        // ---- phi of every K tile as it lands (phase A of a chunk follows at once)
#pragma unroll 1
        for (int p = 0; p < nch && ok; ++p) {
            if (!(ok = wait_bar_warp(prm, abort_flag, &sm.kv_full[p], 0))) break;
            phi_tile_cluster<kVar>(sm.k[p], tid, kScanThreads, prm.N - (c0 + p) * kC, prm);
            fence_proxy_async_smem();
            mbar_arrive(&sm.k_ready[p]);
        }
        // ---- T -> P of chunk p, by group g = warp / 4 for the chunks p with p % 2 == g
        // (T, P and O buffer g): row 32 q + lane of T; key block kb is visible for
        // kb < q, masked on the diagonal for kb == q, zero for kb > q; 16 keys at a time,
        // P half-block hb of key block kb over columns 16 kb + 8 hb .., i.e. over T
        // columns 32 kb + 16 hb .. already read
        const int g = warp >> 2;
        auto t_to_p = [&](int p) -> bool {
            if (!wait_bar_warp(prm, abort_flag, &sm.t_full[g], (p >> 1) & 1)) return false;
            tc_fence_after();
            const uint32_t tb = tl + g * 128;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    uint32_t pk[8];
                    if (kb <= q) {
                        uint32_t t[16];
                        tmem_ld16(tb + kb * 32 + 16 * hb, t);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int jk = 16 * hb + 2 * e;  // key offset within the block
                            pk[e] = (kb < q) ? pack_bf16(__uint_as_float(t[2 * e]), __uint_as_float(t[2 * e + 1]))
                                             : pack_bf16(jk <= lane ? __uint_as_float(t[2 * e]) : 0.f,
                                                         jk + 1 <= lane ? __uint_as_float(t[2 * e + 1]) : 0.f);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) pk[e] = 0u;
                    }
                    tmem_st8(tb + kb * 16 + 8 * hb, pk);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_full[g]);
            return true;
        };
        if (ok && nch > 0) {
            ok = wait_bar_warp(prm, abort_flag, &sm.a_full, 0);
            if (ok) tc_fence_after();
        }
        {
            float run[16], rz = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) run[e] = 0.f;
#pragma unroll
            for (int p = 0; p < kLmax; ++p) {
                if (p < nch && ok) {
                    uint32_t a[16];
                    tmem_ld16(tl + a_col(p) + 16 * h, a);
                    const uint32_t zr = tmem_ld1(tl + a_col(p) + D);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) run[e] += __uint_as_float(a[e]);
                    rz += h == 0 ? __uint_as_float(zr) : 0.f;
                }
                if (p < kLmax - 1) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) cum[p][e] = run[e];
                    cz[p] = rz;
                }
                if (p == nch - 1 && ok) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        xb[(4 * h + e) * D + i] = make_float4(run[4 * e], run[4 * e + 1], run[4 * e + 2], run[4 * e + 3]);
                    if (h == 0) sm.xz[i] = rz;
                }
            }
        }
        if (ok && nch > 0) {
            tc_fence_before();
            mbar_arrive(&sm.a_read);
        }
        if (ok && nch == 0) {  // no chunks: a zero total
#pragma unroll
            for (int e = 0; e < 4; ++e) xb[(4 * h + e) * D + i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (h == 0) sm.xz[i] = 0.f;
        }
        // ---- publish the total to the higher ranks right after phase A
        if (ok) {
            ok = scan_barrier(prm, sm, abort_flag, syncs);  // every thread's part is written
            if (ok && tid == 0)
                for (int r2 = rank + 1; r2 < kG; ++r2) mbar_arrive_remote_release(mapa_shared(smem_u32(&sm.agg_ready), r2));
        }
        if (ok && g < nch) ok = t_to_p(g);
        // ---- scan across the cluster: E = the sum of the lower ranks' segment totals
        float E[16], ez = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) E[e] = 0.f;
        if (ok && rank > 0) ok = wait_bar_warp(prm, abort_flag, &sm.agg_ready, 0, true);
        if (ok) {  // two peers' loads in flight at a time
#pragma unroll
            for (int r0 = 0; r0 < kG - 1; r0 += 2) {
                float4 x[2][4];
                float zx[2] = {0.f, 0.f};
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r2 = r0 + u;
                    if (r2 < rank) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            x[u][e] = ld_dsmem_f4(mapa_shared(smem_u32(xb + (4 * h + e) * D + i), r2));
                        if (h == 0) zx[u] = ld_dsmem_f32(mapa_shared(smem_u32(&sm.xz[i]), r2));
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (r0 + u < rank) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            E[4 * e] += x[u][e].x; E[4 * e + 1] += x[u][e].y;
                            E[4 * e + 2] += x[u][e].z; E[4 * e + 3] += x[u][e].w;
                        }
                        ez += zx[u];
                    }
                }
            }
        }
        // ---- images: chunk p sees E + (running sum after chunk p - 1), written as bf16
        // into the first half of the chunk's K tile and z into the second half, once
        // no MMA reads that K tile any more: phase A is over (the scan read every
        // running sum) and T of chunks 2 j, 2 j + 1 completed (t_done[j], a one-shot
        // barrier).  Pair j then releases the state terms of its chunks (img_ready[j]).
        auto images = [&](int j) -> bool {
            if (!wait_bar_warp(prm, abort_flag, &sm.t_done[j], 0)) return false;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int p = 2 * j + u;
                if (p < nch) {
                    float x[16];
                    float zv = ez;
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = E[e] + (p > 0 ? cum[p > 0 ? p - 1 : 0][e] : 0.f);
                    if (p > 0) zv += cz[p > 0 ? p - 1 : 0];
                    put_img16(sm.k[p], i, 16 * h, x);
                    if (h == 0) put_z_row(sm.k[p] + kSbBytes, i, zv);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.img_ready[j]);
            return true;
        };
        if (ok && nch > 0) ok = images(0);
        if (ok && g + 2 < nch) ok = t_to_p(g + 2);
        if (ok && nch > 2) ok = images(1);
        {
            // ---- O out (this group's chunks): o = O / max(den, eps) as bf16, staged in
            // the chunk's Q tile (no MMA reads it once O is final), written by a TMA store.
            const int row = q * 32 + lane;
            const bool leader = (warp & 3) == 0 && lane == 0;
            const uint64_t pol = l2_policy_evict_first();
            for (int p = g; p < nch && ok; p += 2) {
                const int b = o_buf(p);
                const uint32_t ph = p == 3 ? 1u : 0u;  // buffer 1 holds chunk 1, then chunk 3
                if (!(ok = wait_bar_warp(prm, abort_flag, &sm.o_full[b], ph))) break;
                tc_fence_after();
                const uint32_t to = tl + o_col(b);
                const float den = __uint_as_float(tmem_ld1(to + D)) + __uint_as_float(tmem_ld1(to + D + 1));
                tmem_ld_wait();
                const float inv = (kVar && !prm.normalize) ? 1.f : 1.f / fmaxf(den, prm.eps);
                uint8_t *rowp = sm.q[p] + row * 128;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t a[32];
                    tmem_ld16(to + 32 * hh, *reinterpret_cast<uint32_t(*)[16]>(&a[0]));
                    tmem_ld16(to + 32 * hh + 16, *reinterpret_cast<uint32_t(*)[16]>(&a[16]));
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int cc = 4 * hh + c;
                        *reinterpret_cast<uint4 *>(rowp + ((cc ^ (row & 7)) << 4)) = make_uint4(
                            pack_bf16(__uint_as_float(a[8 * c]) * inv, __uint_as_float(a[8 * c + 1]) * inv),
                            pack_bf16(__uint_as_float(a[8 * c + 2]) * inv, __uint_as_float(a[8 * c + 3]) * inv),
                            pack_bf16(__uint_as_float(a[8 * c + 4]) * inv, __uint_as_float(a[8 * c + 5]) * inv),
                            pack_bf16(__uint_as_float(a[8 * c + 6]) * inv, __uint_as_float(a[8 * c + 7]) * inv));
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&sm.o_staged[b]);
                if (p == 1) {
                    tc_fence_before();
                    mbar_arrive(&sm.o_free);
                }
                bool st_ok = true;
                if (leader && (st_ok = wait_bar(prm, abort_flag, &sm.o_staged[b], ph))) {
                    tma_store_3d_hint(&map_o, sm.q[p], 0, (c0 + p) * kC, bh, pol);
                    tma_store_commit();
                }
                if (!(ok = __all_sync(0xffffffffu, st_ok))) break;
            }
            if (leader) tma_store_wait_all();  // all output stores complete before the CTA exits
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
    // no CTA leaves while a peer may still read its shared memory or arrive on its barriers
    cluster_sync_all();
}

}  // namespace

// bf16, dk = dv = 64, chunk 128, 128 <= N <= 2048 (at most 16 chunks per head), no
// decay; elu + 1 with the normaliser, or a feature-map / normaliser variant.
la_status causal_cluster_tc(const Problem &p)
{
    if (p.dtype != LA_BF16 || p.dk != D || p.dv != D || p.chunk != kC || p.N < kC || p.N > kG * kLmax * kC ||
        p.gamma)
        return LA_ERR_UNSUPPORTED;
    const bool var = !p.var.is_default();
    if ((long long)p.BH * kG > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv, mo;
    la_status st = make_map(&mq, p.q, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mk, p.k, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mv, p.v, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mo, p.o, p.BH, p.N, D);
    if (st != LA_OK) return st;
    Params prm{};
    prm.N = p.N;
    prm.BH = p.BH;
    prm.n_c = ceil_div(p.N, kC);
    prm.L = ceil_div(prm.n_c, kG);
    prm.eps = p.eps;
    prm.wait_ns = test_wait_limit_ns();
    prm.map = p.var.map;
    prm.normalize = p.var.normalize;
    {
        const __nv_bfloat16 c = __float2bfloat16_rn(p.var.shift);
        const uint16_t b = *reinterpret_cast<const uint16_t *>(&c);
        prm.shift2 = (uint32_t)b | ((uint32_t)b << 16);
    }
    auto kern = var ? causal_cluster_kernel<true> : causal_cluster_kernel<false>;
    const int smem = (int)sizeof(Smem);
    st = ensure_smem((const void *)kern, smem);
    if (st != LA_OK) return st;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)(p.BH * kG));
    lc.blockDim = dim3((unsigned)kThreads);
    lc.dynamicSmemBytes = (size_t)smem;
    lc.stream = p.stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kG;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = dependent_launch_allowed(p.stream) ? 2 : 1;
    count_launches();
    return cuda_status(cudaLaunchKernelEx(&lc, kern, mq, mk, mv, mo, prm));
}

la_status tc_cluster_read_status(cudaStream_t s, unsigned *bits)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_cl_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_cl_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // namespace la
