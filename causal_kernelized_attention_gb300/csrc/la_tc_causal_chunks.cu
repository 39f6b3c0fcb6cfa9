// Tensor-core chunk-parallel causal forward, bf16 in / fp32 accumulate,
// dk = dv = 64, chunk C = 128: one work item per chunk, and no chunk waits on
// another chunk of its own CTA.
//
// The chunked form ("Linear Attention", aiwiki.thehackersbrain.dev, listing
// linear_attention_chunked; "Linear Attention -- Math + Variants", Chunkwise
// parallelism): the masked quadratic form inside a chunk, the state
// S = sum phi(k) v^T, z = sum phi(k) across chunks.  The state before chunk c
// is an exclusive prefix over chunks, found by a decoupled look-back over
// per-chunk states:
//
//  * Persistent CTAs take chunk items by ticket, chunk-major (ticket t is chunk
//    t / BH of head t % BH), so the chunks of one head are BH tickets apart.
//  * Per item (b,h,c), on the tensor cores (operands TMA-loaded, 128-byte swizzle):
//      A_c = phi(K_c)^T [V_c | 1]                       the chunk's S and z, fp32 TMEM
//      T   = phi(Q_c) phi(K_c)^T,  P = bf16(tril T)     P written over T in TMEM
//      O   = P [V_c | 1] + phi(Q_c) [E_c | z_c]         E_c: exclusive prefix (bf16 image)
//    o = O / max(rowsum(P) + phi(q) z_c, eps), written by a TMA store.
//  * A_c is published as soon as it is read back (chunk 0's as its inclusive
//    prefix).  The look-back adds, in fp32, the nearest published inclusive prefix
//    I_j and the aggregates A_{j+1} .. A_{c-1}: that is E_c, whose bf16 copy (and z
//    as a bf16 high + low pair) feeds the output MMA; I_c = E_c + A_c is published
//    for the chunks after it.
//  * The MMA thread runs one item ahead: A and T of item n + 1 go to the tensor
//    pipe before the output MMAs of item n, which wait for item n's look-back.
//
// Warp roles (800 threads): warps 0-3 turn T into P (TMEM lane quadrant = warp);
// 4-7 normalise O and store it; 8-9 read A_c back and publish it; 10 tickets and
// TMA loads; 11 the T, P V and output MMAs, and TMEM; 12-19 look-back and the
// state image; 20-23 phi (K first, then Q); 24 the chunk-state MMAs.  Every wait is bounded (Params::wait_ns); on expiry the CTA records
// LA_ERR_TIMEOUT in this file's status word and raises the launch's abort word,
// so that every CTA winds down: each drains its copies and MMAs in flight and
// frees its TMEM before it exits.
#include "la_common.cuh"
#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"

#include <algorithm>

namespace la {
namespace {

using namespace sm100;
using namespace tc;

static __device__ unsigned g_cc_status;

constexpr int D = 64;
constexpr int kThreads = 800;
constexpr int kS = 4;                    // stages: Q, K and V of one chunk each
constexpr int kR = 8;                    // item ring
constexpr uint32_t kTile = kC * D * 2;   // one [128 x 64] bf16 tile: 16 KB
constexpr uint32_t kSbBytes = D * D * 2; // bf16 state image, MN-major for phi(Q) E
constexpr int kOWarp0 = 4, kAggWarp0 = 8, kTmaWarp = 10, kMmaWarp = 11, kLbWarp0 = 12,
              kPhiWarp0 = 20, kAWarp = 24;
constexpr int kPhiThreads = 128, kLbThreads = 256, kAggThreads = 64;
// Readers of a ring entry: 4 T->P warps, 4 O warps, 2 publishing warps, the MMA
// thread, 8 look-back warps, 4 phi warps, the chunk-state MMA thread (one arrival
// per warp).
constexpr uint32_t kRingReaders = 4 + 4 + 2 + 1 + 8 + 4 + 1;
constexpr uint32_t kPublished = 8;       // a published state's counter value
constexpr size_t kStateFloats = (size_t)D * D + D;  // S (thread-major, see add_state), then z
// TMEM columns: T (and P over it) in two buffers of 128, O = [P V | rowsum] +
// phi(Q) [E | z] in two buffers of 80, A_c = [S | z] in 80.
constexpr uint32_t tO = 256, kOStride = 80, tA = 416;
static_assert(tO + 2 * kOStride <= tA && tA + 80 <= 512, "TMEM column groups overlap");
constexpr uint32_t kDrainNs = 100000000u;  // 0.1 s: copies and MMAs in flight always finish

struct Item {
    int bh, c;  // c < 0: no more work
    int t;      // ticket
};

struct alignas(1024) Smem {
    uint8_t q[kS][kTile];
    uint8_t k[kS][kTile];
    uint8_t v[kS][kTile];
    uint8_t img[2][kSbBytes];  // state images E_c (bf16, MN-major), one per item parity
    uint8_t ones[kC * 128];    // column 0 = 1; columns 16(b+1), 16(b+1)+1 = z_hi, z_lo of image b
    uint64_t full[kS], k_ready[kS], phi_done[kS], empty[kS];
    uint64_t item_full[kR], item_empty[kR];
    uint64_t a_full, a_free, drain, drain_a;
    uint64_t t_full[2], p_full[2], pv_done[2], o_full[2], o_free[2], o_staged[2], s_ready[2];
    uint64_t lb_sync;  // the look-back warps' barrier (bounded, unlike bar.sync)
    Item items[kR];
    uint32_t tmem_base;
    int abort;
    int lb_base[2];    // look-back result of an item, by item parity
    int last;
};
static_assert(sizeof(Smem) <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

struct Params {
    float *incl;            // [BH * n_c, kStateFloats] inclusive prefixes I_c (index bh * n_c + c)
    float *agg;             // [BH * n_c, kStateFloats] chunk states A_c
    uint32_t *counter;      // [0] work ticket, [1] CTAs done, [2] abort word of the launch
    uint32_t *incl_cnt;     // [BH * n_c] publish counters of incl
    uint32_t *agg_cnt;      // [BH * n_c] publish counters of agg (right after incl_cnt)
    int N, BH, n_c;
    float eps;
    unsigned long long wait_ns;  // limit of every bounded wait
    long long drop_ticket;       // failure-detection tests: this item never publishes (-1: none)
};

__device__ __forceinline__ bool global_abort(const Params &prm)
{
    return *(volatile uint32_t *)(prm.counter + 2) != 0u;
}
// Gives up the CTA's work; a timed-out wait also records LA_ERR_TIMEOUT and
// raises the launch's abort word, which every other CTA's look-back polls.
__device__ __forceinline__ void give_up(const Params &prm, int *abort_flag, bool timed_out)
{
    *(volatile int *)abort_flag = 1;
    if (timed_out) {
        atomicOr(&g_cc_status, kStatusTimeout);
        atomicExch(prm.counter + 2, 1u);
    }
}

__device__ __forceinline__ bool wait_bar(const Params &prm, int *abort_flag, uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000)) return true;
        if (aborted(abort_flag)) return false;
        if (globaltimer_ns() - t0 > prm.wait_ns) {
            give_up(prm, abort_flag, true);
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bar_warp(const Params &prm, int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, wait_bar(prm, abort_flag, bar, parity));
}
// Waits for a phase that is certain to complete (copies and MMAs in flight), for
// at most kDrainNs, before the CTA frees what they use.
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < kDrainNs) {
    }
}

// The ring entry of iteration `it`, read by one warp (lane 0 frees the entry).
__device__ __forceinline__ bool ring_read(const Params &prm, Smem &sm, int *abort_flag, int it, int lane, Item *out)
{
    const int r = it % kR;
    if (!wait_bar_warp(prm, abort_flag, &sm.item_full[r], (it / kR) & 1)) return false;
    *out = sm.items[r];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.item_empty[r]);
    return true;
}

// z_i of image b as a bf16 high + low pair in columns 16(b+1), 16(b+1)+1 of row i
// of the ones block.
__device__ __forceinline__ void put_z_pair(uint8_t *ones, int i, float zv, int b)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
    const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
    *reinterpret_cast<__nv_bfloat162 *>(ones + sw128_offset(i, 16 * (b + 1))) = __halves2bfloat162(hi, lo);
}

// Row i, columns [16 h, 16 h + 16) of a published state (thread-major layout: the
// float4 of columns 4c..4c+3 of row i at float4 index c * D + i), and z_i for h = 0.
__device__ __forceinline__ void load_part(const float *st, int i, int h, float4 (&x)[4], float &zv)
{
    const float4 *s4 = reinterpret_cast<const float4 *>(st);
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = __ldcg(s4 + (size_t)(4 * h + e) * D + i);
    zv = h == 0 ? __ldcg(st + (size_t)D * D + i) : 0.f;
}
__device__ __forceinline__ void add_part(float (&acc)[16], float &zacc, const float4 (&x)[4], float zv)
{
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        acc[4 * e] += x[e].x; acc[4 * e + 1] += x[e].y; acc[4 * e + 2] += x[e].z; acc[4 * e + 3] += x[e].w;
    }
    zacc += zv;
}
// Row i, columns [col0, col0 + 16) of the bf16 state image (MN-major, 128-byte swizzled, D = 64).
__device__ __forceinline__ void put_sb16(uint8_t *sb, int i, int col0, const float (&x)[16])
{
#pragma unroll
    for (int c8 = 0; c8 < 16; c8 += 8) {
        const int col = col0 + c8;
        *reinterpret_cast<uint4 *>(sb + i * 128 + (((col >> 3) ^ (i & 7)) << 4)) =
            make_uint4(pack_bf16(x[c8], x[c8 + 1]), pack_bf16(x[c8 + 2], x[c8 + 3]), pack_bf16(x[c8 + 4], x[c8 + 5]),
                       pack_bf16(x[c8 + 6], x[c8 + 7]));
    }
}

__global__ void __launch_bounds__(kThreads, 1)
causal_chunks_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                     const Params prm)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // layout assumption of the swizzled tiles
        if (threadIdx.x == 0) atomicOr(&g_cc_status, kStatusTimeout);
        return;
    }
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_items = prm.BH * prm.n_c;
    // The next launch on the stream may start its set-up now; it waits for this
    // grid to complete before it touches global memory.
    griddep_launch_dependents();

    if (warp == kTmaWarp && lane == 0) {
        // Warm L2 with the tiles of tickets blockIdx.x and blockIdx.x + gridDim.x (the
        // first two waves of items, whichever CTAs take them).  A prefetch is only a
        // hint to L2, the point of coherence, so it may run before the grid
        // dependency is resolved.
        for (int t = (int)blockIdx.x; t < n_items && t < 2 * (int)gridDim.x; t += (int)gridDim.x) {
            const int c = t / prm.BH, bh = t % prm.BH;
            tma_prefetch_3d(&map_q, 0, c * kC, bh);
            tma_prefetch_3d(&map_k, 0, c * kC, bh);
            tma_prefetch_3d(&map_v, 0, c * kC, bh);
        }
    }
    if (tid < 128) {
        // ones block: row r holds 1 in column 0 (physical 16-byte chunk r % 8); the z
        // columns are written with each image
        for (int c = tid; c < kC * 8; c += 128) {
            const uint32_t x = (c & 7) == ((c >> 3) & 7) ? 0x3F80u : 0u;
            *reinterpret_cast<uint4 *>(sm.ones + c * 16) = make_uint4(x, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.k_ready[s], kPhiThreads);
            mbar_init(&sm.phi_done[s], kPhiThreads);
            // released by the output store and by the read-back of the chunk state
            mbar_init(&sm.empty[s], 2);
        }
        for (int r = 0; r < kR; ++r) {
            mbar_init(&sm.item_full[r], 1);
            mbar_init(&sm.item_empty[r], kRingReaders);
        }
        mbar_init(&sm.a_full, 1);
        mbar_init(&sm.a_free, kAggThreads);
        mbar_init(&sm.drain, 1);
        mbar_init(&sm.drain_a, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.t_full[b], 1);
            mbar_init(&sm.p_full[b], 128);
            mbar_init(&sm.pv_done[b], 1);
            mbar_init(&sm.o_full[b], 1);
            mbar_init(&sm.o_free[b], 128);
            mbar_init(&sm.o_staged[b], 128);
            mbar_init(&sm.s_ready[b], kLbThreads);
        }
        mbar_init(&sm.lb_sync, kLbThreads);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    // Global memory only after the grids this one depends on are done (the launch
    // before may still be clearing the flags or reading the workspace).
    griddep_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    int *abort_flag = &sm.abort;

    if (warp >= kPhiWarp0 && warp < kAWarp) {
        // ---------------------------------------------------------------- phi warps
        const int t = tid - kPhiWarp0 * 32;
        for (int it = 0;; ++it) {
            Item item;
            if (!ring_read(prm, sm, abort_flag, it, lane, &item) || item.c < 0) break;
            const int s = it % kS;
            if (!wait_bar_warp(prm, abort_flag, &sm.full[s], (it / kS) & 1)) break;
            const int valid = prm.N - item.c * kC;  // rows past the sequence become zeros
            phi_tile<D, kPhiThreads>(sm.k[s], t, valid);
            fence_proxy_async_smem();
            mbar_arrive(&sm.k_ready[s]);  // the chunk-state MMA needs phi(K) only
            phi_tile<D, kPhiThreads>(sm.q[s], t, valid);
            fence_proxy_async_smem();
            mbar_arrive(&sm.phi_done[s]);
        }
    } else if (warp == kAWarp) {
        // ---------------------------------------------------------------- chunk-state MMA
        // A_c = phi(K_c)^T [V_c | 1] as soon as phi(K_c) is done and the publishing
        // warps have read A of the item before: no look-back delays a publication.
        if (lane == 0) {
            const uint32_t id_KV = idesc_bf16_f32(128, D + 16, true, true);  // phi(K)^T [V | 1]
            const uint32_t ones = smem_u32(sm.ones);
            for (int it = 0;; ++it) {
                const int r = it % kR;
                if (!wait_bar(prm, abort_flag, &sm.item_full[r], (it / kR) & 1)) break;
                const Item item = sm.items[r];
                mbar_arrive(&sm.item_empty[r]);
                if (item.c < 0) break;
                const int s = it % kS;
                if (!wait_bar(prm, abort_flag, &sm.k_ready[s], (it / kS) & 1)) break;
                if (it >= 1 && !wait_bar(prm, abort_flag, &sm.a_free, (it - 1) & 1)) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(sm.k[s]), va = smem_u32(sm.v[s]);
                // phi(K)^T is MN-major; its second 64-row block (one tile on) feeds rows
                // 64..127 of A, which nothing reads.
                const uint64_t dkt = mnmajor(ka, 0, kBox), dv = mnmajor(va, 0, ones - va);
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_ss(tmem + tA, dkt + 128 * kk, dv + 128 * kk, id_KV, kk > 0 ? 1u : 0u);
                mma_commit(&sm.a_full);
            }
            // its MMAs complete before TMEM is freed
            mma_commit(&sm.drain_a);
            drain_bar(&sm.drain_a, 0);
        }
    } else if (warp == kTmaWarp) {
        // ---------------------------------------------------------------- tickets + TMA
        if (lane == 0) {
            tma_prefetch_map(&map_q);
            tma_prefetch_map(&map_k);
            tma_prefetch_map(&map_v);
            tma_prefetch_map(&map_o);
            const uint64_t pol = l2_policy_evict_first();  // every tile is read once
            int issued = 0;
            for (int it = 0;; ++it) {
                // A ticket is taken only once its ring entry and stage are free and at
                // most one other load is in flight (the load of item it - 2 has landed):
                // tickets held but not yet loading would unbalance the CTAs.
                const int r = it % kR, s = it % kS;
                if (it >= kR && !wait_bar(prm, abort_flag, &sm.item_empty[r], ((it / kR) - 1) & 1)) break;
                if (it >= kS && !wait_bar(prm, abort_flag, &sm.empty[s], ((it / kS) - 1) & 1)) break;
                if (it >= 2 && !wait_bar(prm, abort_flag, &sm.full[(it - 2) % kS], ((it - 2) / kS) & 1)) break;
                const int t = (int)atomicAdd(prm.counter, 1u);
                Item item{0, -1, t};
                if (t < n_items && !aborted(abort_flag)) {
                    item.c = t / prm.BH;
                    item.bh = t % prm.BH;
                }
                sm.items[r] = item;
                mbar_arrive(&sm.item_full[r]);
                if (item.c < 0) break;
                mbar_arrive_expect_tx(&sm.full[s], 3 * kTile);
                const int row0 = item.c * kC;
                tma_load_3d_hint(sm.q[s], &map_q, &sm.full[s], 0, row0, item.bh, pol);
                tma_load_3d_hint(sm.k[s], &map_k, &sm.full[s], 0, row0, item.bh, pol);
                tma_load_3d_hint(sm.v[s], &map_v, &sm.full[s], 0, row0, item.bh, pol);
                issued = it + 1;
            }
            // No copy may still be writing shared memory when the CTA exits.
            for (int j = max(0, issued - kS); j < issued; ++j) drain_bar(&sm.full[j % kS], (j / kS) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_T = idesc_bf16_f32(128, 128, false, false);   // phi(Q) phi(K)^T
            const uint32_t id_PV = idesc_bf16_f32(128, D + 16, false, true); // P [V | 1] (P in TMEM)
            const uint32_t id_QS = idesc_bf16_f32(128, D + 16, false, true); // phi(Q) [E | z]
            const uint32_t ones = smem_u32(sm.ones);
            // T of item n (stage n % kS) into buffer n % 2 once P V of item n - 2, which
            // read P from it, is done.  (The chunk state A is issued by its own thread.)
            auto issue_T = [&](int n) -> bool {
                const int s = n % kS, b = n & 1;
                if (!wait_bar(prm, abort_flag, &sm.phi_done[s], (n / kS) & 1)) return false;
                const uint32_t qa = smem_u32(sm.q[s]), ka = smem_u32(sm.k[s]);
                if (n >= 2 && !wait_bar(prm, abort_flag, &sm.pv_done[b], ((n - 2) >> 1) & 1)) return false;
                tc_fence_after();
                const uint64_t dq = kmajor(qa, 0), dk = kmajor(ka, 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + b * 128, dq + 2 * kk, dk + 2 * kk, id_T, kk > 0 ? 1u : 0u);
                mma_commit(&sm.t_full[b]);
                return true;
            };
            Item cur;
            bool ok = wait_bar(prm, abort_flag, &sm.item_full[0], 0);
            if (ok) {
                cur = sm.items[0];
                mbar_arrive(&sm.item_empty[0]);
                ok = cur.c >= 0 && issue_T(0);
            }
            for (int n = 0; ok; ++n) {
                const int n1 = n + 1, r1 = n1 % kR;
                if (!(ok = wait_bar(prm, abort_flag, &sm.item_full[r1], (n1 / kR) & 1))) break;
                const Item nx = sm.items[r1];
                mbar_arrive(&sm.item_empty[r1]);
                if (nx.c >= 0 && !(ok = issue_T(n1))) break;
                // outputs of item n: P V into O buffer n % 2 (free once item n - 2's O
                // has been read), then phi(Q) [E | z] once the look-back is done
                const int s = n % kS, b = n & 1;
                if (!(ok = wait_bar(prm, abort_flag, &sm.p_full[b], (n >> 1) & 1))) break;
                if (n >= 2 && !(ok = wait_bar(prm, abort_flag, &sm.o_free[b], ((n - 2) >> 1) & 1))) break;
                tc_fence_after();
                const uint32_t va = smem_u32(sm.v[s]);
                const uint64_t dv = mnmajor(va, 0, ones - va);
                const uint32_t dO = tmem + tO + b * kOStride, dP = tmem + b * 128;
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) mma_ts(dO, dP + kk * 8, dv + 128 * kk, id_PV, kk > 0 ? 1u : 0u);
                mma_commit(&sm.pv_done[b]);
                if (!(ok = wait_bar(prm, abort_flag, &sm.s_ready[b], (n >> 1) & 1))) break;
                tc_fence_after();
                if (cur.c > 0) {
                    const uint32_t sb = smem_u32(sm.img[b]);
                    const uint64_t dsb = mnmajor(sb, 0, ones + 32 * (b + 1) - sb);
                    const uint64_t dq = kmajor(smem_u32(sm.q[s]), 0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) mma_ss(dO, dq + 2 * kk, dsb + 128 * kk, id_QS, 1u);
                }
                mma_commit(&sm.o_full[b]);
                if (nx.c < 0) break;
                cur = nx;
            }
            // all issued MMAs complete before TMEM is freed
            mma_commit(&sm.drain);
            drain_bar(&sm.drain, 0);
        }
    } else if (warp < kOWarp0) {
        // ---------------------------------------------------------------- T -> P (warps 0-3)
        // Row i = 32 quad + lane of T; key block kb (keys 32 kb .. 32 kb + 31) is
        // visible for kb < quad, masked on the diagonal for kb == quad and zero for
        // kb > quad.  P block kb (16 columns of bf16 pairs) is written over columns
        // 16 kb .. 16 kb + 15 of the buffer, which hold T blocks this warp has read
        // already (blocks in increasing order) or never needs.
        const int quad = warp & 3;
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        for (int it = 0;; ++it) {
            Item item;
            if (!ring_read(prm, sm, abort_flag, it, lane, &item) || item.c < 0) break;
            const int b = it & 1;
            if (!wait_bar_warp(prm, abort_flag, &sm.t_full[b], (it >> 1) & 1)) break;
            tc_fence_after();
            const uint32_t tb = tl + b * 128;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                uint32_t pk[16];
                if (kb <= quad) {
                    uint32_t t[32];
                    tmem_ld32(tb + kb * 32, t);
                    tmem_ld_wait();
                    if (kb == quad) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack_bf16(2 * e <= lane ? __uint_as_float(t[2 * e]) : 0.f,
                                              2 * e + 1 <= lane ? __uint_as_float(t[2 * e + 1]) : 0.f);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack_bf16(__uint_as_float(t[2 * e]), __uint_as_float(t[2 * e + 1]));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = 0u;
                }
                tmem_st16(tb + kb * 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_full[b]);
        }
    } else if (warp < kAggWarp0) {
        // ---------------------------------------------------------------- O out (warps 4-7)
        // o = O / max(den, eps), rounded to bf16 and staged (128-byte swizzled) in the
        // Q tile of the item's stage -- no MMA reads Q once O is final -- then written
        // by a TMA store, which clips rows past the end of the sequence.  The stage is
        // released once the store has read it.
        const int quad = warp & 3, i = quad * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        const bool leader = warp == kOWarp0 && lane == 0;
        const uint64_t pol = l2_policy_evict_first();
        int prev_stage = -1;
        for (int it = 0;; ++it) {
            Item item;
            if (!ring_read(prm, sm, abort_flag, it, lane, &item) || item.c < 0) break;
            const int b = it & 1, s = it % kS;
            if (!wait_bar_warp(prm, abort_flag, &sm.o_full[b], (it >> 1) & 1)) break;
            tc_fence_after();
            const uint32_t to = tl + tO + b * kOStride;
            // column D: rowsum(P) + phi(q) z_hi; D + 1: phi(q) z_lo
            const float den = __uint_as_float(tmem_ld1(to + D)) + __uint_as_float(tmem_ld1(to + D + 1));
            tmem_ld_wait();
            const float inv = 1.f / fmaxf(den, prm.eps);
            uint8_t *rowp = sm.q[s] + i * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t a[32];
                tmem_ld16(to + 32 * h, *reinterpret_cast<uint32_t(*)[16]>(&a[0]));
                tmem_ld16(to + 32 * h + 16, *reinterpret_cast<uint32_t(*)[16]>(&a[16]));
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int cc = 4 * h + c;  // 16-byte chunk of the row
                    *reinterpret_cast<uint4 *>(rowp + ((cc ^ (i & 7)) << 4)) = make_uint4(
                        pack_bf16(__uint_as_float(a[8 * c]) * inv, __uint_as_float(a[8 * c + 1]) * inv),
                        pack_bf16(__uint_as_float(a[8 * c + 2]) * inv, __uint_as_float(a[8 * c + 3]) * inv),
                        pack_bf16(__uint_as_float(a[8 * c + 4]) * inv, __uint_as_float(a[8 * c + 5]) * inv),
                        pack_bf16(__uint_as_float(a[8 * c + 6]) * inv, __uint_as_float(a[8 * c + 7]) * inv));
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&sm.o_staged[b]);
            tc_fence_before();
            mbar_arrive(&sm.o_free[b]);
            bool ok = true;
            if (leader && (ok = wait_bar(prm, abort_flag, &sm.o_staged[b], (it >> 1) & 1))) {
                tma_store_3d_hint(&map_o, sm.q[s], 0, item.c * kC, item.bh, pol);
                tma_store_commit();
                // The previous item's store has read its staged O: that stage may be refilled.
                tma_store_wait_read<1>();
                if (prev_stage >= 0) mbar_arrive(&sm.empty[prev_stage]);
                prev_stage = s;
            }
            if (!__all_sync(0xffffffffu, ok)) break;
        }
        if (leader) {
            tma_store_wait_read_all();
            if (prev_stage >= 0) mbar_arrive(&sm.empty[prev_stage]);
            tma_store_wait_all();  // all output stores complete before the CTA exits
        }
    } else if (warp < kTmaWarp) {
        // ---------------------------------------------------------------- publish A_c (warps 8-9)
        // Lanes 0..63 of A hold its 64 rows (key features): warp 8 rows 0-31, warp 9
        // rows 32-63; each thread writes its row in the thread-major state layout.
        // The last chunk of a head has no successor: its state is not published.
        const int quad = warp & 3, i = quad * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        for (int it = 0;; ++it) {
            Item item;
            if (!ring_read(prm, sm, abort_flag, it, lane, &item) || item.c < 0) break;
            if (!wait_bar_warp(prm, abort_flag, &sm.a_full, it & 1)) break;
            tc_fence_after();
            const bool publish = item.c < prm.n_c - 1 && (long long)item.t != prm.drop_ticket;
            const size_t idx = (size_t)item.bh * prm.n_c + item.c;
            float *dst = (item.c == 0 ? prm.incl : prm.agg) + idx * kStateFloats;
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
                uint32_t a[32];
                tmem_ld32(tl + tA + cc, a);
                tmem_ld_wait();
                if (publish) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        d4[(size_t)((cc >> 2) + e) * D + i] =
                            make_float4(__uint_as_float(a[4 * e]), __uint_as_float(a[4 * e + 1]),
                                        __uint_as_float(a[4 * e + 2]), __uint_as_float(a[4 * e + 3]));
                }
            }
            const float zv = __uint_as_float(tmem_ld1(tl + tA + D));
            tmem_ld_wait();
            if (publish) dst[(size_t)D * D + i] = zv;
            tc_fence_before();
            mbar_arrive(&sm.a_free);
            // A_c complete implies its reads of K and V are done: the stage's second release
            if (warp == kAggWarp0 && lane == 0) mbar_arrive(&sm.empty[it % kS]);
            if (publish) {
                // the warp's stores before lane 0's release (two warps, half of kPublished each)
                __syncwarp();
                if (lane == 0) red_release_add_gpu((item.c == 0 ? prm.incl_cnt : prm.agg_cnt) + idx, kPublished / 2);
            }
        }
    } else if (warp >= kLbWarp0 && warp < kPhiWarp0) {
        // ---------------------------------------------------------------- look-back (warps 12-15)
        // Thread lt owns state row i = lt % 64 and columns [16 h, 16 h + 16), h = lt / 64
        // (h = 0 also z_i).  The group's first warp finds, among the 32 chunks before
        // c, the nearest published inclusive prefix I_j with every aggregate after it
        // published; all four warps then add them.
        const int lt = tid - kLbWarp0 * 32, i = lt & 63, h = lt >> 6;  // h: columns 16 h .. 16 h + 15
        uint32_t syncs = 0;  // completed uses of lb_sync
        for (int it = 0;; ++it) {
            Item item;
            if (!ring_read(prm, sm, abort_flag, it, lane, &item) || item.c < 0) break;
            const int b = it & 1;
            // image b was last read by the output MMAs of item it - 2 (this wait also
            // keeps s_ready[b] at most one phase ahead of the MMA thread)
            if (it >= 2 && !wait_bar_warp(prm, abort_flag, &sm.o_full[b], ((it - 2) >> 1) & 1)) break;
            const bool last = item.c == prm.n_c - 1;
            const size_t head0 = (size_t)item.bh * prm.n_c;
            if (item.c > 0) {
                if (warp == kLbWarp0) {
                    int base = -1;
                    const uint64_t t0 = globaltimer_ns();
                    while (true) {
                        const int j = item.c - 1 - lane;
                        uint32_t ci = 0, ca = 0;
                        if (j >= 0) {
                            ci = ld_acquire_gpu(prm.incl_cnt + head0 + j);
                            ca = ld_acquire_gpu(prm.agg_cnt + head0 + j);
                        }
                        // this chunk's own aggregate (read for I_c below)
                        const uint32_t own = (last || lane != 0) ? kPublished : ld_acquire_gpu(prm.agg_cnt + head0 + item.c);
                        const bool own_ok = __shfl_sync(0xffffffffu, own, 0) == kPublished;
                        const unsigned inc = __ballot_sync(0xffffffffu, ci == kPublished);
                        const unsigned avail = __ballot_sync(0xffffffffu, ci == kPublished || ca == kPublished);
                        const int first = inc ? __ffs(inc) - 1 : 32;  // nearest inclusive prefix
                        const unsigned need = first >= 32 ? 0xffffffffu : ((1u << first) - 1u);
                        if (first < 32 && (avail & need) == need && own_ok) {
                            base = item.c - 1 - first;
                            break;
                        }
                        if (aborted(abort_flag) || global_abort(prm)) {
                            if (lane == 0) give_up(prm, abort_flag, false);
                            break;
                        }
                        if (globaltimer_ns() - t0 > prm.wait_ns) {
                            if (lane == 0) give_up(prm, abort_flag, true);
                            break;
                        }
                    }
                    if (lane == 0) sm.lb_base[b] = base;
                }
                // Every thread of the group reads lb_base[b] after this barrier; the slot
                // is next written for item it + 2, after every thread has passed the
                // barrier of item it + 1.  A bounded wait: a warp that gave up earlier
                // never arrives.
                mbar_arrive(&sm.lb_sync);
                const bool synced = wait_bar_warp(prm, abort_flag, &sm.lb_sync, syncs & 1);
                ++syncs;
                const int base = synced ? sm.lb_base[b] : -1;
                if (base < 0) break;  // gave up
                // States of the look-back: I_base, then A_{base+1} .. A_{c-1} (their sum is
                // E_c), then A_c (for I_c).  Two states' loads are in flight per round trip.
                auto st_ptr = [&](int j) -> const float * {
                    return (j == base ? prm.incl : prm.agg) + (head0 + j) * kStateFloats;
                };
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.f;
                float zacc = 0.f;
                int j = base;
                for (; j + 1 < item.c; j += 2) {
                    float4 x0[4], x1[4];
                    float z0, z1;
                    load_part(st_ptr(j), i, h, x0, z0);
                    load_part(st_ptr(j + 1), i, h, x1, z1);
                    add_part(acc, zacc, x0, z0);
                    add_part(acc, zacc, x1, z1);
                }
                // the last state of E_c (if any) and A_c in the same round trip
                float4 xe[4], xo[4];
                float ze = 0.f, zo = 0.f;
                const bool e_left = j < item.c;
                if (e_left) load_part(st_ptr(j), i, h, xe, ze);
                if (!last) load_part(prm.agg + (head0 + item.c) * kStateFloats, i, h, xo, zo);
                if (e_left) add_part(acc, zacc, xe, ze);
                put_sb16(sm.img[b], i, 16 * h, acc);
                if (h == 0) put_z_pair(sm.ones, i, zacc, b);
                fence_proxy_async_smem();
                if (!last) {  // I_c = E_c + A_c for the chunks after this one
                    add_part(acc, zacc, xo, zo);
                    float *dst = prm.incl + (head0 + item.c) * kStateFloats;
                    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        d4[(size_t)(4 * h + e) * D + i] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2],
                                                                      acc[4 * e + 3]);
                    if (h == 0) dst[(size_t)D * D + i] = zacc;
                }
            }
            mbar_arrive(&sm.s_ready[b]);
            if (item.c > 0 && !last) {
                __syncwarp();
                if (lane == 0) red_release_add_gpu(prm.incl_cnt + head0 + item.c, 1u);
            }
        }
    }

    tc_fence_before();
    __threadfence();  // this CTA's flag traffic is done before it counts itself finished
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
    // The last CTA to finish leaves the ticket, the counters, the abort word and
    // every publish counter of this launch at zero, ready for the next launch.
    if (tid == 0) sm.last = atom_add_acq_rel_gpu(prm.counter + 1, 1u) == gridDim.x - 1;
    __syncthreads();
    if (sm.last) {
        for (int x = tid; x < 2 * n_items; x += kThreads) prm.incl_cnt[x] = 0u;  // incl_cnt then agg_cnt
        if (tid == 0) {
            prm.counter[0] = 0u;
            prm.counter[1] = 0u;
            prm.counter[2] = 0u;
        }
    }
}

}  // namespace

// Chosen by causal_tc for bf16, dk = dv = 64, chunk 128, N >= 128, elu + 1 with the
// normaliser and no decay, when there are enough heads that the chunks of one head
// in flight at a time fit the look-back window.
la_status causal_chunks_tc(const Problem &p)
{
    if (p.dtype != LA_BF16 || p.dk != D || p.dv != D || p.chunk != kC || p.N < kC || p.gamma ||
        !p.var.is_default())
        return LA_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv, mo;
    la_status st = make_map(&mq, p.q, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mk, p.k, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mv, p.v, p.BH, p.N, D);
    if (st == LA_OK) st = make_map(&mo, p.o, p.BH, p.N, D);
    if (st != LA_OK) return st;

    const int n_c = ceil_div(p.N, kC);
    const long long items = (long long)p.BH * n_c;
    if (items > 0x3fffffffLL) return LA_ERR_UNSUPPORTED;
    const size_t flag_bytes = ((16 + (size_t)items * 8) + 255) / 256 * 256;
    const size_t state_bytes = 2 * (size_t)items * kStateFloats * 4;

    // Flags and states from the stream's workspaces (flags already zero) when they
    // can serve the call, else from per-call scratch (flags cleared by a memset).
    void *ws = nullptr, *data = nullptr;
    st = flag_workspace(p.stream, flag_bytes, &ws);
    if (st != LA_OK && st != LA_ERR_UNSUPPORTED) return st;
    st = data_workspace(p.stream, state_bytes, &data);
    if (st != LA_OK && st != LA_ERR_UNSUPPORTED) return st;
    const size_t own_flags = ws ? 0 : flag_bytes;
    const size_t own_state = data ? 0 : state_bytes;
    Scratch scratch;
    if (own_flags + own_state > 0) {
        st = scratch.alloc(own_flags + own_state, p.stream);
        if (st != LA_OK) return st;
    }
    uint8_t *base = (uint8_t *)scratch.ptr;
    uint8_t *flags = ws ? (uint8_t *)ws : base;
    uint8_t *states = data ? (uint8_t *)data : base + own_flags;
    if (!ws) {
        cudaError_t e = cudaMemsetAsync(flags, 0, flag_bytes, p.stream);
        count_launches();
        if (e != cudaSuccess) return cuda_status(e);
    }

    Params prm{};
    prm.counter = (uint32_t *)flags;
    prm.incl_cnt = (uint32_t *)(flags + 16);
    prm.agg_cnt = prm.incl_cnt + items;
    prm.incl = (float *)states;
    prm.agg = prm.incl + (size_t)items * kStateFloats;
    prm.N = p.N;
    prm.BH = p.BH;
    prm.n_c = n_c;
    prm.eps = p.eps;
    prm.wait_ns = test_wait_limit_ns();
    prm.drop_ticket = test_drop_ticket();

    const int smem = (int)sizeof(Smem);
    st = ensure_smem((const void *)causal_chunks_kernel, smem);
    if (st != LA_OK) return st;
    const unsigned grid = (unsigned)std::min<long long>(items, sm_count());
    count_launches();
    return launch_dependent(causal_chunks_kernel, grid, kThreads, smem, p.stream, mq, mk, mv, mo, prm);
}

la_status tc_chunks_read_status(cudaStream_t s, unsigned *bits)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_cc_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_cc_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // namespace la
