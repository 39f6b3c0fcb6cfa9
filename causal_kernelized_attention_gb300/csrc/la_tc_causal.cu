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
//  * Phase B: the exclusive scan of the chunk states across segments, in fp32,
//    by decoupled look-back: publish A_g, sum the predecessors' aggregates back
//    to the nearest published inclusive prefix (bounded waits), publish
//    P_g = P_{g-1} + A_g, and load P_{g-1} as the running state.
//  * Phase C: sweep the segment's chunks.  Per chunk c, on the tensor cores:
//      T   = phi(Q_c) phi(K_c)^T                         (fp32, TMEM)
//      P   = bf16(tril(T))                               (TMEM, written by threads)
//      O   = P V_c + phi(Q_c) bf16(S)                    (fp32, TMEM)
//      rs  = P 1,  qz = phi(Q_c) (z_hi + z_lo)           (denominator terms)
//      S  += phi(K_c)^T V_c,  z += phi(K_c)^T 1          (running state, fp32 TMEM)
//    o = O / max(rs + qz, eps), written as bf16.
//
// Warp roles (576 threads): warps 0-7 apply phi in shared memory; warp 8 issues
// TMA loads; warp 9 issues MMAs and owns TMEM; warps 10-13 turn T into P; warps
// 14-17 normalise O and refresh the bf16 copy of S; warps 10-17 run phase B.  Waiting
// threads sleep on the mbarrier (suspend-time hint) rather than spin, so they
// leave issue slots to the working warps.  Every wait is bounded by
// %globaltimer; on expiry the CTA records LA_ERR_TIMEOUT in its status word,
// abandons its work, drains its in-flight copies and MMAs, and frees its TMEM.
#include "la_common.cuh"
#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"
#include "la_tc_pad.cuh"

#include <algorithm>
#include <mutex>
#include <unordered_map>

namespace la {
namespace {

using namespace sm100;
using namespace tc;

static __device__ unsigned g_tc_status;

constexpr int kThreads = 576;
constexpr int kPhiThreads = 256;         // warps 0-7
// Epilogue warps access the TMEM lane quadrant warp % 4, so each group of four
// consecutive warps covers all 128 lanes.
constexpr int kTmaWarp = 8, kMmaWarp = 9, kEpiPWarp0 = 10, kEpiOWarp0 = 14;
// Per-segment publish counters: each of the 8 phase-B warps adds 1 (with release
// semantics) once its part of a state is stored; kPublished means complete, and
// kPoison or more marks a segment whose CTA gave up.
constexpr uint32_t kPublished = 8, kPoison = 1u << 20;
constexpr int kMaxShortSegs = 32;  // segments per head in short-sequence mode
constexpr int kChunkKernelMinHeads = 16;  // B*H from which d = 64 runs the chunk-parallel kernel
constexpr int kClusterKernelMaxN = 2048;  // sequences up to which d = 64 runs the cluster kernel

// Row sums and z ride on the tensor cores in one of two ways:
//  * fused (D = 64): the B operand of P V and of the state update is [V | 1] and
//    that of phi(Q) S is [S_bf16 | z]: one N = D + 16 MMA whose second 64-wide
//    block (an LBO away) is the ones block (column 0 = 1) or a z block (columns
//    0 and 1 = z_hi, z_lo), so result column D holds the row sum or z.  The ones
//    block's rows use only column 0, so the two z blocks (one per bf16 S copy) live
//    in its columns 16.. and 32..: a start address 32 or 64 bytes on;
//  * separate (D = 128, no room for those blocks): N = 16 MMAs against W, a
//    [16 rows x 128] bf16 K-major operand (two 1 KB blocks of 8 rows; rows 8..15 of
//    its descriptor alias into the next 2 KB, the S copy, and feed only unread
//    columns).  Row 0 = ones, rows 1 and 2 = the high and low bf16 parts of z.
template <int D>
struct Cfg {
    static constexpr bool kFused = D == 64;
    static constexpr int kStages = D == 128 ? 2 : 4;
    static constexpr uint32_t kTileBytes = kC * D * 2;
    static constexpr uint32_t kSbBytes = D * D * 2;   // bf16 copy of S, MN-major for the phi(Q) S MMA
    // aux: fused = two bf16 S copies, then the ones block (128 rows) holding the two z
    // blocks; separate = W, then the S copy
    static constexpr uint32_t kW = 0;
    static constexpr uint32_t kSb = kFused ? 0 : 2048;
    static constexpr uint32_t kOnes = 2 * kSbBytes;
    static constexpr uint32_t kAuxBytes = kFused ? kOnes + kC * 128 : kSb + kSbBytes;
    // TMEM columns.  Fused: P and O have two buffers each (kPStride, kOStride
    // apart), O and S are D + 16 wide, z in column D of S.  Separate: one P and one
    // O buffer, row sums and phi(q) z in their own 16-column groups, z at tZ.
    static constexpr uint32_t tT = 0, tP = 128, tRS = 192, tQZ = 208;
    static constexpr uint32_t kPStride = kFused ? 64 : 0;
    static constexpr uint32_t tO = 256, kOStride = kFused ? D + 16 : 0;
    static constexpr uint32_t tS = kFused ? 416 : 256 + D;
    static constexpr uint32_t tZ = kFused ? tS + D : 224;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kFused ? (tP + 2 * kPStride <= tO && tO + 2 * kOStride <= tS && tS + D + 16 <= kTmemCols &&
                            tS % 32 == 0 && kOStride % 16 == 0)
                         : (tP + 64 <= tRS && tRS + 16 <= tQZ && tQZ + 16 <= tO && tO + D <= tS &&
                            tS + D <= kTmemCols),
                  "TMEM column groups overlap");
};

template <int D>
struct alignas(1024) Smem {
    uint8_t q[Cfg<D>::kStages][Cfg<D>::kTileBytes];
    uint8_t k[Cfg<D>::kStages][Cfg<D>::kTileBytes];
    uint8_t v[Cfg<D>::kStages][Cfg<D>::kTileBytes];
    uint8_t aux[Cfg<D>::kAuxBytes];
    uint64_t full[Cfg<D>::kStages], phi_done[Cfg<D>::kStages], empty[Cfg<D>::kStages];
    uint64_t ostore[Cfg<D>::kStages];  // the O tile staged in slot s has been read by its TMA store
    uint64_t t_full, t_free, s_full, s_ready, agg_ready, drain;
    uint64_t p_full[2];  // per P buffer (the separate layout uses buffer 0)
    uint64_t o_full[2], o_free[2];  // per O buffer (the separate layout uses buffer 0)
    uint64_t o_staged[2];           // all 128 rows of the buffer's O tile are staged in shared memory
    float gp[32 + kC];              // decayed state: gp[32 + d] = gamma^d for d in [0, C), 0 for d < 0
    uint32_t tmem_base;
    int ticket;
    int abort;
    int lb_base;  // look-back result
    int last;     // this CTA finished last: it clears the flags for the next launch
};

static_assert(sizeof(Smem<128>) <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
static_assert(sizeof(Smem<64>) <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

struct Params {
    uint16_t *o;            // bf16 output [BH, N, D]
    float *incl;            // [BH, G, D*D + D] inclusive prefixes (S then z; thread-major, see add_state)
    float *agg;             // [BH, G, D*D + D] segment aggregates (same layout)
    uint32_t *incl_cnt;     // [BH, G] publish counters of incl
    uint32_t *agg_cnt;      // [BH, G] publish counters of agg
    uint32_t *counter;      // work ticket; counter[1] counts finished CTAs
    int N, BH, G, L, n_chunks;
    float eps;
    // Short sequences: segment g of every head is chunks [bounds[g], bounds[g + 1]);
    // it sums its own prefix (chunks before bounds[g]) in phase A, so no segment
    // waits on another (no ticket, scan or flags).  0: the scan over L-chunk segments.
    int short_mode;
    int bounds[kMaxShortSegs + 1];
    // Decayed state: gamma[bh % H] per head (device memory); unused otherwise.
    const float *gamma;
    int H;
    // Feature-map variant (kVar): LA_PHI_* map with shift; normalize 0: o = phi(q)^T S.
    int map;
    float shift;
    int normalize;
    // Feature widths (multiples of 8, at most D): q, k carry dk columns, v, o dv;
    // the tiles' columns past them are zero (see zero_cols).
    int dk, dv;
};

__device__ __forceinline__ bool wait_bar(int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return tc::wait_bar(&g_tc_status, abort_flag, bar, parity);
}
__device__ __forceinline__ bool wait_bar_warp(int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return tc::wait_bar_warp(&g_tc_status, abort_flag, bar, parity);
}

// z_i as a bf16 high + low pair: fused, in columns 16(b+1) and 16(b+1)+1 of row i
// of the ones block (z block b); separate, in rows 1 and 2 of W.
template <int D>
__device__ __forceinline__ void set_z(uint8_t *aux, int i, float zv, int b)
{
    if constexpr (Cfg<D>::kFused) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
        const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat162 *>(aux + Cfg<D>::kOnes + sw128_offset(i, 16 * (b + 1))) =
            __halves2bfloat162(hi, lo);
    } else {
        put_z(aux + Cfg<D>::kW, i, zv);
    }
}
// bf16 S copy b (fused: b = target chunk % 2; separate: the single copy).
template <int D>
__device__ __forceinline__ uint8_t *sb_copy(uint8_t *aux, int b)
{
    return aux + Cfg<D>::kSb + (Cfg<D>::kFused ? b * Cfg<D>::kSbBytes : 0);
}

// Chunk of job j: phase-A jobs walk chunks [a0, a0 + nA) backwards -- the segment
// itself (scan: a0 = c0), so that phase C, which walks it forwards, starts with the
// K and V tiles read most recently (the likeliest still in L2), or the chunks
// before it (short sequences: a0 = 0); a sum, so its order is free.
__device__ __forceinline__ int job_chunk(int j, int nA, int a0, int c0)
{
    return j < nA ? a0 + (nA - 1 - j) : c0 + (j - nA);
}

// The work of ticket t: segment g of head bh is chunks [c0, c0 + nch); phase A sums
// the nA chunks from a0 (scan: the segment itself when it has a successor;
// short sequences: the chunks before it, its exclusive prefix).
struct Seg {
    int g, bh, c0, nch, a0, nA;
    bool has_next;  // scan mode: a later segment reads this one's aggregate
};
__device__ __forceinline__ Seg segment_of(const Params &prm, int t)
{
    Seg r;
    r.g = t / prm.BH;
    r.bh = t % prm.BH;
    if (prm.short_mode) {
        r.c0 = prm.bounds[r.g];
        r.nch = prm.bounds[r.g + 1] - r.c0;
        r.a0 = 0;
        r.nA = r.c0;
        r.has_next = false;
    } else {
        r.c0 = r.g * prm.L;
        r.nch = min(prm.L, prm.n_chunks - r.c0);
        r.has_next = r.g < prm.G - 1;
        r.a0 = r.c0;
        r.nA = r.has_next ? r.nch : 0;
    }
    return r;
}

// S += phi(K_c)^T [V_c | 1] (fused) or S += phi(K_c)^T V_c and z += phi(K_c)^T 1.
// phi(K_c)^T is MN-major with its second dk block one box on (D = 64: the next
// tile, whose rows 64..127 of the result are never read).
template <int D>
__device__ __forceinline__ void issue_state_update(uint32_t tmem, uint32_t ka, uint32_t va, uint32_t lbo_v,
                                                   uint32_t w_addr, uint32_t id_KV, uint32_t id_KW, bool first)
{
#pragma unroll
    for (int kk = 0; kk < kC / 16; ++kk) {
        const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
        mma_ss(tmem + Cfg<D>::tS, mnmajor(ka, kk, kBox), mnmajor(va, kk, lbo_v), id_KV, acc);
        if constexpr (!Cfg<D>::kFused)
            mma_ss(tmem + Cfg<D>::tZ, mnmajor(ka, kk, kBox), wdesc(w_addr, kk), id_KW, acc);
    }
}

// The bf16 copy of S (and z) for the next chunk, from S_acc, once s_full completes.
// The bf16 copy (and z) of the state for chunk cj + 1, from S_acc once chunk cj's
// state update is done (s_full).  Fused: into copy (cj + 1) % 2, the caller signals
// through p_full; separate: the single copy, then s_ready.
// Decayed state: S_acc and z are also scaled in place by gC = gamma^C, ready for the
// next chunk's update S = gamma^C S + sum_j gamma^(C-1-j) phi(k_j) [v_j | 1]^T.
template <int D, bool kDecay>
__device__ __forceinline__ bool refresh_state(Smem<D> &sm, int *abort_flag, uint32_t tl, int i, bool row_ok, int cj,
                                              float gC)
{
    using CF = Cfg<D>;
    if (!wait_bar_warp(abort_flag, &sm.s_full, cj & 1)) return false;
    tc_fence_after();
#pragma unroll 1
    for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t a[64];
        tmem_ld32(tl + CF::tS + cc * 64, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
        tmem_ld32(tl + CF::tS + cc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&a[32]));
        tmem_ld_wait();
        if (row_ok) {
            float x[32];
            to_floats(&a[0], x);
            put_sb<D>(sb_copy<D>(sm.aux, (cj + 1) & 1), i, cc * 64, x);
            to_floats(&a[32], x);
            put_sb<D>(sb_copy<D>(sm.aux, (cj + 1) & 1), i, cc * 64 + 32, x);
        }
        if constexpr (kDecay) {
#pragma unroll
            for (int e = 0; e < 64; ++e) a[e] = __float_as_uint(__uint_as_float(a[e]) * gC);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                tmem_st16(tl + CF::tS + cc * 64 + 16 * q4, *reinterpret_cast<const uint32_t(*)[16]>(&a[16 * q4]));
        }
    }
    const float zv = __uint_as_float(tmem_ld1(tl + CF::tZ));
    tmem_ld_wait();
    if (row_ok) set_z<D>(sm.aux, i, zv, (cj + 1) & 1);
    if constexpr (kDecay) {
        tmem_st1(tl + CF::tZ, __float_as_uint(zv * gC));
        tmem_st_wait();
    }
    fence_proxy_async_smem();
    if constexpr (!CF::kFused) {
        tc_fence_before();
        mbar_arrive(&sm.s_ready);
    }
    return true;
}

// T -> P for the key blocks in `blocks` (bit b = keys 32b..32b+31) of this warp's
// 32 query rows (32*quad .. 32*quad+31): block b is entirely visible for b < quad,
// masked on the diagonal for b == quad, and entirely masked (zeros, no TMEM read)
// for b > quad.  When t_free is given, it is arrived on once T has been read.
// Decayed state: key b of query row a is also weighted by gp[32 + a - b] = gamma^(a - b)
// (0 for b > a: the table's first 32 entries).
template <int D, bool kDecay>
__device__ __forceinline__ void convert_tp(uint32_t tl, uint32_t tPb, int quad, int lane, unsigned blocks,
                                           uint64_t *t_free, const float *gp)
{
    uint32_t t[32];
    uint32_t pk[16];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        if (!((blocks >> b) & 1u)) continue;
        if (b <= quad) {
            tmem_ld32(tl + Cfg<D>::tT + b * 32, t);
            tmem_ld_wait();
            if constexpr (kDecay) {
                const float *w = gp + 32 + 32 * (quad - b) + lane;  // at a - (first key of the block)
#pragma unroll
                for (int e = 0; e < 32; ++e) t[e] = __float_as_uint(__uint_as_float(t[e]) * w[-e]);
            }
            if (b == quad) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int jk = 2 * e;  // key offset within the diagonal block
                    pk[e] = pack_bf16(jk <= lane ? __uint_as_float(t[2 * e]) : 0.f,
                                      jk + 1 <= lane ? __uint_as_float(t[2 * e + 1]) : 0.f);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(__uint_as_float(t[2 * e]), __uint_as_float(t[2 * e + 1]));
            }
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
        }
        if (t_free && b == 3) {  // all of T that this warp reads has been read
            tc_fence_before();
            mbar_arrive(t_free);
        }
        tmem_st16(tl + tPb + b * 16, pk);
    }
    tmem_st_wait();
}

// add_state, plus z_i of the same state (issued with it) when want_z.
template <int D>
__device__ __forceinline__ void add_state_z(float (&acc)[32], float &zacc, const float *state, int cg0, int i,
                                            bool want_z)
{
    const float zv = want_z ? __ldcg(state + (size_t)D * D + i) : 0.f;
    add_state<D>(acc, state, cg0, i);
    zacc += zv;
}
// add_state_z with the state weighted by w (decayed state: gamma^(tokens since it ended)).
template <int D>
__device__ __forceinline__ void add_state_zw(float (&acc)[32], float &zacc, const float *state, int cg0, int i,
                                             bool want_z, float w)
{
    const float zv = want_z ? __ldcg(state + (size_t)D * D + i) : 0.f;
    const float4 *s4 = reinterpret_cast<const float4 *>(state);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float4 x = __ldcg(s4 + (size_t)(cg0 + e) * D + i);
        acc[4 * e] += w * x.x; acc[4 * e + 1] += w * x.y; acc[4 * e + 2] += w * x.z; acc[4 * e + 3] += w * x.w;
    }
    zacc += w * zv;
}

template <int D, bool kDecay, bool kVar>
__global__ void __launch_bounds__(576, 1)
causal_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                 const Params prm)
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
    uint8_t *const sb = sb_copy<D>(sm.aux, 0);  // phase B writes the state for the first chunk here
    // The next launch on the stream may start its set-up now; it waits for this
    // grid to complete before it touches global memory.
    griddep_launch_dependents();

    // The work ticket is taken first (once the grids this one depends on are done:
    // the launch before may still be clearing the flags), its latency hidden behind
    // the set-up.  A CTA that waits on an earlier ticket waits on a running CTA: no
    // other CTA of this library fits on an SM beside one of this kernel (shared
    // memory), so the TMEM allocation below can only wait on other kernels' CTAs,
    // which never wait on it.  Every other thread reaches global memory after the
    // set-up barrier, hence after this thread's griddep_wait.
    // (Short sequences: no segment waits on another, so the segment is blockIdx.x
    // and no ticket is taken.)
    int my_ticket = 0;
    if (tid == 0) {
        griddep_wait();
        my_ticket = prm.short_mode ? (int)blockIdx.x : (int)atomicAdd(prm.counter, 1u);
    }
    if (warp == kTmaWarp && lane == 0) {
        // While the ticket is out: warm L2 with the first tiles of segment blockIdx.x.
        // Every segment belongs to exactly one CTA, which reads these tiles first,
        // whichever CTA draws that ticket.  A prefetch is only a hint to L2 (the point
        // of coherence), so it may run before the grid dependency is resolved.
        const Seg ps = segment_of(prm, (int)blockIdx.x);
        for (int x = 0; x < min(ps.nA + ps.nch, S); ++x) {
            const int row0 = job_chunk(x, ps.nA, ps.a0, ps.c0) * kC;
#pragma unroll
            for (int b = 0; b < D / 64; ++b) {  // (boxes past a width hold no data)
                if (64 * b < prm.dk) {
                    if (x >= ps.nA) tma_prefetch_3d(&map_q, 64 * b, row0, ps.bh);
                    tma_prefetch_3d(&map_k, 64 * b, row0, ps.bh);
                }
                if (64 * b < prm.dv) tma_prefetch_3d(&map_v, 64 * b, row0, ps.bh);
            }
        }
    }

    if (tid < 128) {
        if constexpr (CF::kFused) {
            // ones block: row r holds 1 in column 0 (physical 16-byte chunk r % 8); z block zero
            for (int c = tid; c < kC * 8; c += 128) {
                const uint32_t x = (c & 7) == ((c >> 3) & 7) ? 0x3F80u : 0u;
                *reinterpret_cast<uint4 *>(sm.aux + CF::kOnes + c * 16) = make_uint4(x, 0u, 0u, 0u);
            }
        } else {  // W: row 0 ones, everything else zero (rows 1, 2 get z in phase B)
            const int blk = tid >> 6, within = tid & 63;
            const uint32_t val = (within < 8) ? 0x3F803F80u : 0u;  // first 128 bytes of a block = row 0
            *reinterpret_cast<uint4 *>(sm.aux + CF::kW + blk * 1024 + within * 16) = make_uint4(val, val, val, val);
        }
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            // 512 arrivals: phi threads and epilogue threads share the K tiles of
            // phase A; for phase-C jobs each phi thread arrives with a count of 2.
            mbar_init(&sm.phi_done[s], 2 * kPhiThreads);
            mbar_init(&sm.empty[s], 1);
            mbar_init(&sm.ostore[s], 1);
        }
        mbar_init(&sm.t_full, 1);
        mbar_init(&sm.t_free, 128);
        for (int b = 0; b < 2; ++b)
            mbar_init(&sm.p_full[b], CF::kFused ? 256 : 128);  // fused: the T->P and the O warps convert
        for (int ob = 0; ob < 2; ++ob) {
            mbar_init(&sm.o_full[ob], 1);
            mbar_init(&sm.o_free[ob], 128);
            mbar_init(&sm.o_staged[ob], 128);
        }
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
    if (tid == 0) sm.ticket = my_ticket;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const Seg seg = segment_of(prm, sm.ticket);
    const int g = seg.g, bh = seg.bh, c0 = seg.c0, nch = seg.nch, a0 = seg.a0, nA = seg.nA;
    const bool has_next = seg.has_next;  // scan: publishing only when a successor exists
    const int total = nA + nch;
    const uint32_t tmem = sm.tmem_base;
    int *abort_flag = &sm.abort;
    // Decayed state: lg = log2(gamma) of this head; phase A weights token t of its
    // range by gamma^(eA - t), eA = the range's last token.
    const float lg = kDecay ? log2f(__ldg(prm.gamma + bh % prm.H)) : 0.f;
    const int eA = (a0 + nA) * kC - 1;

    if (warp < kPhiThreads / 32) {
        // ---------------------------------------------------------------- phi warps
        for (int j = 0; j < total; ++j) {
            const int s = j % S, r = j / S;
            if (!wait_bar(abort_flag, &sm.full[s], r & 1)) break;
            const bool isC = j >= nA;
            const int chunk = job_chunk(j, nA, a0, c0);
            const int valid = prm.N - chunk * kC;
            if (isC) {
                phi_tile<D, kPhiThreads, false, kVar>(sm.k[s], tid, valid, 0.f, 0, prm.map, prm.shift);
                if (prm.dk < D) zero_cols<D>(sm.k[s], tid, kPhiThreads, prm.dk);
                phi_tile<D, kPhiThreads, false, kVar>(sm.q[s], tid, valid, 0.f, 0, prm.map, prm.shift);
            } else {  // the other half: epilogue warps
                phi_tile<D, 2 * kPhiThreads, kDecay, kVar>(sm.k[s], tid, valid, lg, eA - chunk * kC, prm.map, prm.shift);
                if (prm.dk < D) zero_cols<D>(sm.k[s], tid, 2 * kPhiThreads, prm.dk);
            }
            fence_proxy_async_smem();
            if (isC)
                mbar_arrive_cnt(&sm.phi_done[s], 2);
            else
                mbar_arrive(&sm.phi_done[s]);
        }
    } else if (warp == kTmaWarp) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_map(&map_q);
            tma_prefetch_map(&map_k);
            tma_prefetch_map(&map_v);
            tma_prefetch_map(&map_o);
            // All tiles are loaded evict-first.  (Keeping phase A's K and V with
            // evict-last for their second read in phase C measured slower on long
            // sequences: 1 MB of them per CTA outgrows L2 across the GPU anyway.)
            const uint64_t pol_first = l2_policy_evict_first();
            int issued = 0;
            for (int j = 0; j < total; ++j) {
                const int s = j % S, r = j / S;
                if (r > 0 && !wait_bar(abort_flag, &sm.empty[s], (r - 1) & 1)) break;
                if (j - S >= nA) {  // the previous user of slot s was a C-job: its Q buffer staged O
                    const int first_c = nA + ((s - nA % S) % S + S) % S;
                    const int k = (j - S - first_c) / S;  // index of that C-job among slot s's C-jobs
                    if (!wait_bar(abort_flag, &sm.ostore[s], k & 1)) break;
                }
                const bool isC = j >= nA;
                const int row0 = job_chunk(j, nA, a0, c0) * kC;
                mbar_arrive_expect_tx(&sm.full[s], (isC ? 3u : 2u) * CF::kTileBytes);
#pragma unroll
                for (int b = 0; b < D / 64; ++b) {
                    if (isC) tma_load_3d_hint(sm.q[s] + b * kBox, &map_q, &sm.full[s], 64 * b, row0, bh, pol_first);
                    tma_load_3d_hint(sm.k[s] + b * kBox, &map_k, &sm.full[s], 64 * b, row0, bh, pol_first);
                    tma_load_3d_hint(sm.v[s] + b * kBox, &map_v, &sm.full[s], 64 * b, row0, bh, pol_first);
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
            constexpr int NE = CF::kFused ? D + 16 : D;  // N of the MMAs against V or S
            const uint32_t id_T = idesc_bf16_f32(128, 128, false, false);   // phi(Q) phi(K)^T
            const uint32_t id_PV = idesc_bf16_f32(128, NE, false, true);    // P [V | 1] (P in TMEM)
            const uint32_t id_QS = idesc_bf16_f32(128, NE, false, true);    // phi(Q) [S_bf16 | z]
            const uint32_t id_KV = idesc_bf16_f32(128, NE, true, true);     // phi(K)^T [V | 1]
            const uint32_t id_W = idesc_bf16_f32(128, 16, false, false);    // x W^T (A K-major or TMEM)
            const uint32_t id_KW = idesc_bf16_f32(128, 16, true, false);    // phi(K)^T W^T
            const uint32_t aux = smem_u32(sm.aux);
            const uint32_t w_addr = aux + CF::kW, sb_addr = aux + CF::kSb, ones_addr = aux + CF::kOnes;
            // Second 64-wide block of [S_bf16 | z] (fused: z block b, in the ones block
            // 32(b+1) bytes on) or of the S copy itself (D = 128).
            const uint32_t lbo_sb = D * 128;
            bool ok = true;
            // phase A: aggregate state of the segment
            for (int ja = 0; ja < nA && ok; ++ja) {
                const int s = ja % S, r = ja / S;
                if (!(ok = wait_bar(abort_flag, &sm.phi_done[s], r & 1))) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(sm.k[s]), va = smem_u32(sm.v[s]);
                const uint32_t lbo_v = CF::kFused ? ones_addr - va : kBox;  // [V | 1] or V's second box
                issue_state_update<D>(tmem, ka, va, lbo_v, w_addr, id_KV, id_KW, ja == 0);
                mma_commit(&sm.empty[s]);
            }
            if (ok && nA > 0) mma_commit(&sm.agg_ready);
            // phase C: outputs
            if constexpr (CF::kFused) {
                // Software-pipelined over chunks.  Chunk c waits for p_full(c), which also
                // stands for "T(c) read, the bf16 state for chunk c in place, phi of
                // chunk c + 1 done" (the T -> P warps wait for those), then issues:
                //   S_acc += phi(K_c)^T [V_c | 1]  (the state for chunk c + 1: first, so
                //            that the T -> P warps can make its bf16 copy at once),
                //   T(c + 1) (into the T buffer they convert next, into the other P buffer),
                //   O(c) = P(c) [V_c | 1] + phi(Q_c)[S | z]  (O buffer c % 2, copy c % 2).
                // p_full(c + 1) can then complete while O(c) is still in the tensor pipe.
                // The descriptors of one chunk differ by constant steps of the start address.
                if (nch > 0) {
                    const int s0 = nA % S;
                    if ((ok = wait_bar(abort_flag, &sm.phi_done[s0], (nA / S) & 1))) {
                        tc_fence_after();
                        const uint64_t dq = kmajor(smem_u32(sm.q[s0]), 0), dk = kmajor(smem_u32(sm.k[s0]), 0);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tmem + CF::tT, dq + 2 * kk, dk + 2 * kk, id_T, kk > 0 ? 1u : 0u);
                        mma_commit(&sm.t_full);
                    }
                }
                for (int cj = 0; cj < nch && ok; ++cj) {
                    const int j = nA + cj, s = j % S, ob = cj & 1;
                    const uint32_t dO = tmem + CF::tO + ob * CF::kOStride;
                    const uint32_t dP = tmem + CF::tP + ob * CF::kPStride;
                    const uint32_t va = smem_u32(sm.v[s]);
                    const uint64_t dv = mnmajor(va, 0, ones_addr - va);           // [V | 1], + 128 per kk
                    const uint32_t sbc = sb_addr + ob * CF::kSbBytes;
                    const uint64_t dsb = mnmajor(sbc, 0, ones_addr + 32 * (ob + 1) - sbc);  // [S | z]
                    const uint64_t dqc = kmajor(smem_u32(sm.q[s]), 0);          // + 2 per kk
                    // p_full(cj) also stands for "O buffer ob free": every O warp finishes
                    // reading O of chunk cj - 2 (load wait, fence, its o_free arrival) before
                    // it converts T(cj) and arrives on p_full(cj), so no o_free wait here
                    // (a completed mbarrier wait still costs the issuer ~250 cycles).
                    if (!(ok = wait_bar(abort_flag, &sm.p_full[ob], (cj >> 1) & 1))) break;
                    tc_fence_after();
                    if (cj < nch - 1) {
                        const uint64_t dkt = mnmajor(smem_u32(sm.k[s]), 0, kBox);  // phi(K)^T, + 128 per kk
#pragma unroll
                        for (int kk = 0; kk < kC / 16; ++kk)
                            mma_ss(tmem + CF::tS, dkt + 128 * kk, dv + 128 * kk, id_KV, 1u);
                        mma_commit(&sm.s_full);
                    }
                    if (cj + 1 < nch) {
                        const int s1 = (j + 1) % S;
                        const uint64_t dq1 = kmajor(smem_u32(sm.q[s1]), 0), dk1 = kmajor(smem_u32(sm.k[s1]), 0);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(tmem + CF::tT, dq1 + 2 * kk, dk1 + 2 * kk, id_T, kk > 0 ? 1u : 0u);
                        mma_commit(&sm.t_full);
                    }
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_ts(dO, dP + kk * 8, dv + 128 * kk, id_PV, kk > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(dO, dqc + 2 * kk, dsb + 128 * kk, id_QS, 1u);
                    mma_commit(&sm.o_full[ob]);
                    if (j + S < total) mma_commit(&sm.empty[s]);  // only a stage that is refilled
                }
            } else {
                // D = 128: per chunk T, phi(Q) S and its z term, P V and the row sums, then
                // the state update -- O first, since its store frees the stage.
                for (int cj = 0; cj < nch && ok; ++cj) {
                    const int j = nA + cj, s = j % S, r = j / S;
                    if (!(ok = wait_bar(abort_flag, &sm.phi_done[s], r & 1))) break;
                    tc_fence_after();
                    if (cj > 0 && !(ok = wait_bar(abort_flag, &sm.t_free, (cj - 1) & 1))) break;
                    tc_fence_after();
                    const uint32_t qa = smem_u32(sm.q[s]), ka = smem_u32(sm.k[s]), va = smem_u32(sm.v[s]);
                    const uint32_t lbo_v = kBox;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + CF::tT, kmajor(qa, kk), kmajor(ka, kk), id_T, kk > 0 ? 1u : 0u);
                    mma_commit(&sm.t_full);
                    if (cj > 0 && !(ok = wait_bar(abort_flag, &sm.o_free[0], (cj - 1) & 1))) break;
                    if (!(ok = wait_bar(abort_flag, &sm.s_ready, cj & 1))) break;
                    tc_fence_after();
                    if constexpr (kDecay) {  // phi(Q) of the chunk is scaled before p_full
                        if (!(ok = wait_bar(abort_flag, &sm.p_full[0], cj & 1))) break;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        mma_ss(tmem + CF::tO, kmajor(qa, kk), mnmajor(sb_addr, kk, lbo_sb), id_QS, kk > 0 ? 1u : 0u);
                        mma_ss(tmem + CF::tQZ, kmajor(qa, kk), wdesc(w_addr, kk), id_W, kk > 0 ? 1u : 0u);
                    }
                    if constexpr (!kDecay) {
                        if (!(ok = wait_bar(abort_flag, &sm.p_full[0], cj & 1))) break;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk) {
                        mma_ts(tmem + CF::tO, tmem + CF::tP + kk * 8, mnmajor(va, kk, lbo_v), id_PV, 1u);
                        mma_ts(tmem + CF::tRS, tmem + CF::tP + kk * 8, wdesc(w_addr, kk), id_W, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&sm.o_full[0]);
                    if (cj < nch - 1) {
                        issue_state_update<D>(tmem, ka, va, lbo_v, w_addr, id_KV, id_KW, false);
                        mma_commit(&sm.s_full);
                    }
                    mma_commit(&sm.empty[s]);
                }
            }
            // all issued MMAs complete before TMEM is freed
            mma_commit(&sm.drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&sm.drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else if (warp >= kEpiPWarp0) {
        // ---------------------------------------------------------------- epilogue warps 10-17
        const int quad = warp & 3, i = quad * 32 + lane;  // query row / state row = TMEM lane
        const bool is_o = warp >= kEpiOWarp0;              // warps 14-17: O and state refresh
        const int gtid = (warp - kEpiPWarp0) * 32 + lane;  // 0..255
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        const bool row_ok = i < D;

        // ---- phase B: exclusive prefix of this segment by decoupled look-back.
        // A segment with a successor publishes its aggregate as soon as phase A
        // is done -- segment 0's aggregate is its inclusive prefix and is published
        // as such -- and its inclusive prefix after this CTA has set up its own
        // running state.  A CTA sums the aggregates of its predecessors back to the
        // nearest published inclusive prefix.  Each thread owns state row i and the
        // columns [col0, col0 + D/2).
        // Phase A: the epilogue warps are otherwise idle, so they apply phi to the
        // second half of each K tile (units 256..511).
        if (kDecay && gtid < 32 + kC) sm.gp[gtid] = gtid < 32 ? 0.f : pow_decay(lg, gtid - 32);  // read after phase B's barrier
        const float gC = pow_decay(lg, kC);
        for (int j = 0; j < nA; ++j) {
            const int s = j % S, r = j / S;
            if (!wait_bar(abort_flag, &sm.full[s], r & 1)) break;
            const int chunk = job_chunk(j, nA, a0, c0);
            phi_tile<D, 2 * kPhiThreads, kDecay, kVar>(sm.k[s], kPhiThreads + gtid, prm.N - chunk * kC, lg,
                                                      eA - chunk * kC, prm.map, prm.shift);
            if (prm.dk < D) zero_cols<D>(sm.k[s], kPhiThreads + gtid, 2 * kPhiThreads, prm.dk);
            fence_proxy_async_smem();
            mbar_arrive(&sm.phi_done[s]);
        }

        constexpr int kHalf = D / 2;
        const int col0 = is_o ? kHalf : 0;
        const size_t seg_floats = (size_t)D * D + D;
        const size_t head0 = (size_t)bh * prm.G, my = head0 + g;
        bool have_agg = false;
        if (nA > 0) have_agg = wait_bar_warp(abort_flag, &sm.agg_ready, 0);
        tc_fence_after();
        if (prm.short_mode) {
            // Short sequences: phase A left the exclusive prefix in S_acc (zero-filled
            // here when the segment starts the sequence); its bf16 copy and z for the
            // first chunk.
#pragma unroll 1
            for (int cc = 0; cc < kHalf; cc += 32) {
                float acc[32];
                if (have_agg) {
                    uint32_t a[32];
                    tmem_ld32(tl + CF::tS + col0 + cc, a);
                    tmem_ld_wait();
                    to_floats(a, acc);
                    if constexpr (kDecay) {  // S_acc = gamma^C S for the first chunk's update
#pragma unroll
                        for (int e = 0; e < 32; ++e) a[e] = __float_as_uint(acc[e] * gC);
                        tmem_st16(tl + CF::tS + col0 + cc, *reinterpret_cast<const uint32_t(*)[16]>(&a[0]));
                        tmem_st16(tl + CF::tS + col0 + cc + 16, *reinterpret_cast<const uint32_t(*)[16]>(&a[16]));
                    }
                } else {
                    const uint32_t zero16[16] = {};
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
                    tmem_st16(tl + CF::tS + col0 + cc, zero16);
                    tmem_st16(tl + CF::tS + col0 + cc + 16, zero16);
                }
                if (row_ok) put_sb<D>(sb, i, col0 + cc, acc);
            }
            if (!is_o) {  // z, by the warps of the first column half
                float za = 0.f;
                if (have_agg) {
                    za = __uint_as_float(tmem_ld1(tl + CF::tZ));
                    tmem_ld_wait();
                    if constexpr (kDecay) tmem_st1(tl + CF::tZ, __float_as_uint(za * gC));
                } else {
                    tmem_st1(tl + CF::tZ, 0u);
                }
                if (row_ok) set_z<D>(sm.aux, i, za, 0);
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            tc_fence_before();
            if (is_o) mbar_arrive(&sm.s_ready);  // sb and S_acc of both halves are in place
        } else {
            if (has_next) {
                float *dst = (g == 0 ? prm.incl : prm.agg) + my * seg_floats;
                if (have_agg) {
    #pragma unroll 1
                    for (int cc = 0; cc < kHalf; cc += 32) {
                        uint32_t a[32];
                        tmem_ld32(tl + CF::tS + col0 + cc, a);
                        tmem_ld_wait();
                        if (row_ok) {
                            float4 *d4 = reinterpret_cast<float4 *>(dst);
                            const int cg0 = (col0 + cc) >> 2;
    #pragma unroll
                            for (int e = 0; e < 8; ++e)
                                d4[(size_t)(cg0 + e) * D + i] =
                                    make_float4(__uint_as_float(a[4 * e]), __uint_as_float(a[4 * e + 1]),
                                                __uint_as_float(a[4 * e + 2]), __uint_as_float(a[4 * e + 3]));
                        }
                    }
                    if (!is_o) {
                        const float za = __uint_as_float(tmem_ld1(tl + CF::tZ));
                        tmem_ld_wait();
                        if (row_ok) dst[(size_t)D * D + i] = za;
                    }
                }
                __syncwarp();
                if (lane == 0) red_release_add_gpu((g == 0 ? prm.incl_cnt : prm.agg_cnt) + my, have_agg ? 1u : kPoison);
            }
            if (gtid < 32) {
                // One warp reads the counters of up to 32 predecessors per round.
                int base = -1;
                bool bad = false;
                if (g > 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (true) {
                        const int j = g - 1 - lane;
                        uint32_t ci = 0, ca = 0;
                        if (j >= 0) {
                            ci = ld_acquire_gpu(prm.incl_cnt + head0 + j);
                            ca = ld_acquire_gpu(prm.agg_cnt + head0 + j);
                        }
                        const unsigned inc = __ballot_sync(0xffffffffu, ci == kPublished);
                        const unsigned avail = __ballot_sync(0xffffffffu, ci == kPublished || ca == kPublished);
                        const unsigned poison = __ballot_sync(0xffffffffu, ci >= kPoison || ca >= kPoison);
                        const int first = inc ? __ffs(inc) - 1 : 32;  // nearest inclusive prefix
                        const unsigned need = first >= 32 ? 0xffffffffu : ((1u << first) - 1u);
                        if ((poison & (need | (first < 32 ? (1u << first) : 0u))) != 0u) {
                            bad = true;
                            break;
                        }
                        if (first < 32 && (avail & need) == need) {
                            base = g - 1 - first;
                            break;
                        }
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            if (lane == 0) atomicOr(&g_tc_status, kStatusTimeout);
                            bad = true;
                            break;
                        }
                    }
                }
                if (lane == 0) {
                    sm.lb_base = base;
                    if (bad) *(volatile int *)abort_flag = 1;
                }
            }
            named_bar_sync(1, 256);
            const int base = sm.lb_base;
            const bool use_prev = g > 0 && !aborted(abort_flag);
            float *incl_out = (has_next && g > 0) ? prm.incl + my * seg_floats : nullptr;
            float zacc = 0.f;  // z prefix, summed by the warps of the first column half with their first block
    #pragma unroll 1
            for (int cc = 0; cc < kHalf; cc += 32) {
                float acc[32];
    #pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] = 0.f;
                const int cg0 = (col0 + cc) >> 2;
                const bool want_z = !is_o && cc == 0;
                if (use_prev && row_ok) {
                    if constexpr (kDecay) {
                        // the state that ended with segment j is weighted by gamma^((g-1-j) L C)
                        const int seg_tokens = prm.L * kC;
                        if (base >= 0)
                            add_state_zw<D>(acc, zacc, prm.incl + (head0 + base) * seg_floats, cg0, i, want_z,
                                            pow_decay(lg, (g - 1 - base) * seg_tokens));
                        for (int j = base + 1; j < g; ++j)
                            add_state_zw<D>(acc, zacc, prm.agg + (head0 + j) * seg_floats, cg0, i, want_z,
                                            pow_decay(lg, (g - 1 - j) * seg_tokens));
                    } else {
                        if (base >= 0) add_state_z<D>(acc, zacc, prm.incl + (head0 + base) * seg_floats, cg0, i, want_z);
                        int j = base + 1;
                        for (; j + 1 < g; j += 2) {  // two states per round trip
                            add_state_z<D>(acc, zacc, prm.agg + (head0 + j) * seg_floats, cg0, i, want_z);
                            add_state_z<D>(acc, zacc, prm.agg + (head0 + j + 1) * seg_floats, cg0, i, want_z);
                        }
                        if (j < g) add_state_z<D>(acc, zacc, prm.agg + (head0 + j) * seg_floats, cg0, i, want_z);
                    }
                }
                // decayed state: this segment's own aggregate ends L C tokens after acc's state
                const float gL = kDecay ? pow_decay(lg, prm.L * kC) : 1.f;
                if (incl_out) {
                    uint32_t a[32];
                    if (have_agg) {
                        tmem_ld32(tl + CF::tS + col0 + cc, a);
                        tmem_ld_wait();
                    } else {
    #pragma unroll
                        for (int e = 0; e < 32; ++e) a[e] = 0u;
                    }
                    if (row_ok) {
                        float4 *d4 = reinterpret_cast<float4 *>(incl_out);
    #pragma unroll
                        for (int e = 0; e < 8; ++e)
                            d4[(size_t)(cg0 + e) * D + i] = make_float4(gL * acc[4 * e] + __uint_as_float(a[4 * e]),
                                                gL * acc[4 * e + 1] + __uint_as_float(a[4 * e + 1]),
                                                gL * acc[4 * e + 2] + __uint_as_float(a[4 * e + 2]),
                                                gL * acc[4 * e + 3] + __uint_as_float(a[4 * e + 3]));
                    }
                }
                if constexpr (kDecay) {  // S_acc = gamma^C S for the first chunk's update
                    if (row_ok) put_sb<D>(sb, i, col0 + cc, acc);
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] *= gC;
                    tmem_st16(tl + CF::tS + col0 + cc, *reinterpret_cast<const uint32_t(*)[16]>(&acc[0]));
                    tmem_st16(tl + CF::tS + col0 + cc + 16, *reinterpret_cast<const uint32_t(*)[16]>(&acc[16]));
                } else {
                    tmem_st16(tl + CF::tS + col0 + cc, *reinterpret_cast<const uint32_t(*)[16]>(&acc[0]));
                    tmem_st16(tl + CF::tS + col0 + cc + 16, *reinterpret_cast<const uint32_t(*)[16]>(&acc[16]));
                    if (row_ok) put_sb<D>(sb, i, col0 + cc, acc);
                }
            }
            if (!is_o) {  // z, by the warps of the first column half
                if (incl_out) {
                    float za = 0.f;
                    if (have_agg) {
                        za = __uint_as_float(tmem_ld1(tl + CF::tZ));
                        tmem_ld_wait();
                    }
                    if (row_ok) incl_out[(size_t)D * D + i] = (kDecay ? pow_decay(lg, prm.L * kC) : 1.f) * zacc + za;
                }
                tmem_st1(tl + CF::tZ, __float_as_uint(kDecay ? zacc * gC : zacc));
                if (row_ok) set_z<D>(sm.aux, i, zacc, 0);
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            tc_fence_before();
            if (is_o) mbar_arrive(&sm.s_ready);  // sb and S_acc of both halves are in place
            if (incl_out) {  // publish the inclusive prefix (its stores were issued above)
                __syncwarp();
                if (lane == 0)
                    red_release_add_gpu(prm.incl_cnt + my, (have_agg && !aborted(abort_flag)) ? 1u : kPoison);
            }
        }

        if (!is_o) {
            // ------------------------------------------------------------ T -> P
            for (int cj = 0; cj < nch; ++cj) {
                if constexpr (CF::kFused) {
                    // P buffer cj % 2 and bf16 copy cj % 2 were last read by chunk cj - 2's
                    // MMAs (o_full of that chunk); then the bf16 state for chunk cj (made
                    // once chunk cj - 1's state update is done, which the MMA thread issues
                    // before T(cj); the first chunk's came from phase B).
                    if (cj >= 2 && !wait_bar_warp(abort_flag, &sm.o_full[cj & 1], ((cj >> 1) - 1) & 1)) break;
                    if (cj >= 1 && !refresh_state<D, kDecay>(sm, abort_flag, tl, i, row_ok, cj - 1, gC)) break;
                }
                if (!wait_bar_warp(abort_flag, &sm.t_full, cj & 1)) break;
                const uint32_t tPb = CF::tP + (cj & 1) * CF::kPStride;
                tc_fence_after();
                if constexpr (kDecay) {
                    // T(cj) is done with phi(Q), phi(K) of this chunk: row a of phi(Q) takes
                    // gamma^(a+1) for phi(Q)[S | z], row j of phi(K) gamma^(C-1-j) for the
                    // state update (D = 64: the O warps scale phi(K)).
                    const int s = (nA + cj) % S;
                    scale_row<D>(sm.q[s], i, pow_decay(lg, i + 1));
                    if constexpr (!CF::kFused) scale_row<D>(sm.k[s], i, pow_decay(lg, kC - 1 - i));
                    fence_proxy_async_smem();
                }
                // Fused layout: key blocks 0 and 3 here, 1 and 2 by the O warp of the same
                // lane quadrant (no warp reads more than two blocks); D = 128: all four.
                if constexpr (CF::kFused)
                    convert_tp<D, kDecay>(tl, tPb, quad, lane, 0x9u, nullptr, sm.gp);
                else
                    convert_tp<D, kDecay>(tl, tPb, quad, lane, 0xFu, &sm.t_free, sm.gp);
                if constexpr (CF::kFused) {  // p_full(cj) also stands for phi of chunk cj + 1
                    if (cj + 1 < nch && !wait_bar_warp(abort_flag, &sm.phi_done[(nA + cj + 1) % S],
                                                       ((nA + cj + 1) / S) & 1))
                        break;
                }
                tc_fence_before();
                mbar_arrive(&sm.p_full[CF::kFused ? (cj & 1) : 0]);
            }
        } else {
            // ------------------------------------------------------------ O out (, state refresh)
            // O is staged (bf16, 128-byte swizzled boxes) in the Q buffer of its own
            // slot -- Q is no longer read once O is final -- and written by a TMA
            // store, which clips rows past the end of the sequence.  With D = 128 these
            // warps then make the bf16 copy of the next chunk's state (after O, whose
            // store frees the stage); the fused layout has the T -> P warps do it, and
            // these warps convert key blocks 1 and 2 of each T, which is ready (t_full
            // of chunk it) before O of the chunk before it (o_full of chunk it - 1).
            const bool leader = (warp == kEpiOWarp0 && lane == 0);
            for (int it = 0; it < nch + (CF::kFused ? 1 : 0); ++it) {
                if constexpr (CF::kFused) {
                    if (it < nch) {
                        if (!wait_bar_warp(abort_flag, &sm.t_full, it & 1)) break;
                        tc_fence_after();
                        if constexpr (kDecay) {  // phi(K) row j of this chunk: gamma^(C-1-j)
                            scale_row<D>(sm.k[(nA + it) % S], i, pow_decay(lg, kC - 1 - i));
                            fence_proxy_async_smem();
                        }
                        // (P buffer it % 2 is free: these warps saw o_full of chunk it - 2
                        // in the previous iteration)
                        convert_tp<D, kDecay>(tl, CF::tP + (it & 1) * CF::kPStride, quad, lane, 0x6u, nullptr, sm.gp);
                        tc_fence_before();
                        mbar_arrive(&sm.p_full[it & 1]);
                    }
                    if (it == 0) continue;
                }
                const int cj = CF::kFused ? it - 1 : it;
                const int s = (nA + cj) % S;
                const int ob = CF::kFused ? (cj & 1) : 0;                       // O buffer
                const uint32_t opar = CF::kFused ? ((cj >> 1) & 1) : (cj & 1);  // its phase
                const uint32_t tOb = CF::tO + ob * CF::kOStride;
                if (!wait_bar_warp(abort_flag, &sm.o_full[ob], opar)) break;
                tc_fence_after();
                float den;
                {
                    uint32_t dn[32];
                    if constexpr (CF::kFused) {
                        // column D: rs + phi(q) z_hi; D + 1: phi(q) z_lo (16-column loads: O
                        // buffer 1 starts on a 16-column boundary)
                        tmem_ld16(tl + tOb + D, *reinterpret_cast<uint32_t(*)[16]>(&dn[0]));
                        tmem_ld_wait();
                        den = __uint_as_float(dn[0]) + __uint_as_float(dn[1]);
                    } else {
                        tmem_ld32(tl + CF::tRS, dn);  // columns: rs[0..15], qz[0..15]
                        tmem_ld_wait();
                        den = __uint_as_float(dn[0]) + __uint_as_float(dn[17]) + __uint_as_float(dn[18]);
                    }
                }
                const float inv = (kVar && !prm.normalize) ? 1.f : 1.f / fmaxf(den, prm.eps);
#pragma unroll 1
                for (int cc = 0; cc < D / 64 && 64 * cc < prm.dv; ++cc) {  // (columns past dv are not stored)
                    uint32_t a[64];
                    if constexpr (CF::kFused) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            tmem_ld16(tl + tOb + cc * 64 + 16 * q4, *reinterpret_cast<uint32_t(*)[16]>(&a[16 * q4]));
                    } else {
                        tmem_ld32(tl + tOb + cc * 64, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
                        tmem_ld32(tl + tOb + cc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&a[32]));
                    }
                    tmem_ld_wait();
                    uint8_t *rowp = sm.q[s] + cc * kBox + i * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(rowp + ((c ^ (i & 7)) << 4)) = make_uint4(
                            pack_bf16(__uint_as_float(a[8 * c]) * inv, __uint_as_float(a[8 * c + 1]) * inv),
                            pack_bf16(__uint_as_float(a[8 * c + 2]) * inv, __uint_as_float(a[8 * c + 3]) * inv),
                            pack_bf16(__uint_as_float(a[8 * c + 4]) * inv, __uint_as_float(a[8 * c + 5]) * inv),
                            pack_bf16(__uint_as_float(a[8 * c + 6]) * inv, __uint_as_float(a[8 * c + 7]) * inv));
                }
                // o_staged before o_free: the next o_full of this buffer needs every
                // thread's o_free (D = 128) or every thread's p_full arrival for that
                // chunk, which follows this iteration (fused), so no thread can arrive on
                // o_staged[ob] for that chunk while another has yet to arrive for this one.
                fence_proxy_async_smem();
                mbar_arrive(&sm.o_staged[ob]);
                tc_fence_before();
                mbar_arrive(&sm.o_free[ob]);
                if (leader && wait_bar(abort_flag, &sm.o_staged[ob], opar)) {
                    const uint64_t pol_once = l2_policy_evict_first();
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc)
                        if (64 * cc < prm.dv)
                            tma_store_3d_hint(&map_o, sm.q[s] + cc * kBox, 64 * cc, (c0 + cj) * kC, bh, pol_once);
                    tma_store_commit();
                }
                if (!CF::kFused && cj < nch - 1 && !refresh_state<D, kDecay>(sm, abort_flag, tl, i, row_ok, cj, gC))
                    break;
                if (leader) {  // slot s may be refilled once the store has read the staged O
                    tma_store_wait_read_all();
                    mbar_arrive(&sm.ostore[s]);
                }
            }
            if (leader) tma_store_wait_all();  // all output stores complete before the CTA exits
        }
    }

    tc_fence_before();
    __threadfence();  // this CTA's flag traffic is done before it counts itself finished
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, CF::kTmemCols);
    // The last CTA to finish leaves the ticket, the counter and every publish flag
    // of this launch at zero, ready for the next launch on the same flags.  (Short
    // sequences touch no flag.)
    if (prm.short_mode) return;
    if (tid == 0) sm.last = atom_add_acq_rel_gpu(prm.counter + 1, 1u) == gridDim.x - 1;
    __syncthreads();
    if (sm.last) {
        const int n = 2 * prm.BH * prm.G;  // incl_cnt then agg_cnt
        for (int x = tid; x < n; x += kThreads) prm.incl_cnt[x] = 0u;
        if (tid == 0) {
            prm.counter[0] = 0u;
            prm.counter[1] = 0u;
        }
    }
}

// ------------------------------------------------------------------ host side
template <int D, bool kDecay, bool kVar>
la_status launch(const Problem &p)
{
    CUtensorMap mq, mk, mv, mo;
    la_status st = make_map(&mq, p.q, p.BH, p.N, p.dk);
    if (st == LA_OK) st = make_map(&mk, p.k, p.BH, p.N, p.dk);
    if (st == LA_OK) st = make_map(&mv, p.v, p.BH, p.N, p.dv);
    if (st == LA_OK) st = make_map(&mo, p.o, p.BH, p.N, p.dv);
    if (st != LA_OK) return st;

    const int n_chunks = ceil_div(p.N, kC);
    const long long work = (long long)p.BH * n_chunks;
    const int n_sm = sm_count();
    // Scan: chunks per segment enough to fill the GPU, at most 16 (longer segments
    // mean fewer scan steps; the K, V re-read of phase C should still hit L2).
    int L = (int)std::min<long long>(16, std::max<long long>(1, (work + n_sm - 1) / n_sm));
    int G = ceil_div(n_chunks, L);
    // Short sequences: segments that sum their own prefix instead (no scan), with
    // boundaries that balance a segment's cost -- a prefix chunk counts 1 (8 MMAs),
    // an output chunk 3 (24 MMAs and the T -> P hand-off) -- over at most one wave.
    // Taken when that balanced cost is below the scan's: 4 per chunk of its
    // segments plus about 8 for the publish / look-back / state set-up round trips.
    int bounds[kMaxShortSegs + 1] = {};
    int short_G = 0, short_T = 0;
    if (n_chunks <= kMaxShortSegs) {
        const int gmax = std::max(1, std::min(n_chunks, n_sm / std::max(1, p.BH)));
        for (int T = 3;; ++T) {
            int c = 0, gg = 0;
            while (c < n_chunks && gg < gmax) {
                const int len = (T - c) / 3;  // output chunks this segment affords
                if (len < 1) break;           // T too small
                c = std::min(n_chunks, c + len);
                bounds[++gg] = c;
            }
            if (c >= n_chunks) {
                short_G = gg;
                short_T = T;
                break;
            }
        }
    }
    const bool short_mode = short_G > 0 && short_T <= 4 * L + 8;
    if (short_mode) {
        G = short_G;
        L = 0;
    }
    const size_t items = (size_t)p.BH * G;
    const size_t flag_bytes = ((items * 8 + 16) + 255) / 256 * 256;
    const size_t state_bytes = !short_mode && G > 1 ? 2 * items * ((size_t)D * D + D) * 4 : 0;

    // Flags and published states from the stream's workspaces (flags already zero)
    // when they can serve the call, else from per-call scratch (flags cleared by a
    // memset).  With both workspaces, consecutive calls on the stream are kernel
    // after kernel, which lets a launch overlap the tail of the one before it.
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
    prm.o = (uint16_t *)p.o;
    prm.counter = (uint32_t *)flags;
    prm.incl_cnt = (uint32_t *)(flags + 16);
    prm.agg_cnt = prm.incl_cnt + items;
    prm.incl = (float *)states;
    prm.agg = prm.incl + (G > 1 ? items * ((size_t)D * D + D) : 0);
    prm.N = p.N;
    prm.BH = p.BH;
    prm.G = G;
    prm.L = L;
    prm.n_chunks = n_chunks;
    prm.eps = p.eps;
    prm.short_mode = short_mode ? 1 : 0;
    for (int x = 0; x <= G && short_mode; ++x) prm.bounds[x] = bounds[x];
    prm.gamma = p.gamma;
    prm.H = p.H;
    prm.map = p.var.map;
    prm.shift = p.var.shift;
    prm.normalize = p.var.normalize;
    prm.dk = p.dk;
    prm.dv = p.dv;

    const int smem = (int)sizeof(Smem<D>);
    auto kern = causal_tc_kernel<D, kDecay, kVar>;
    st = ensure_smem((const void *)kern, smem);
    if (st != LA_OK) return st;
    count_launches();
    return launch_dependent(kern, (unsigned)items, kThreads, smem, p.stream, mq, mk, mv, mo, prm);
}

}  // namespace

la_status causal_tc(const Problem &p_in)
{
    // The chunked form computes the same function for every chunk length (only the
    // order of the roundings differs), so a request for chunks of 64 runs here too,
    // with the tensor-core kernels' 128-token tiles.
    if (p_in.chunk != 64 && p_in.chunk != kC) return LA_ERR_UNSUPPORTED;
    Problem p = p_in;
    p.chunk = kC;
    if (p.dtype != LA_BF16 || p.N < kC) return LA_ERR_UNSUPPORTED;
    const bool var = !p.var.is_default();
    if (p.dk != p.dv || (p.dk != 64 && p.dk != 128)) {
        // Other widths (multiples of 8 up to 128, dk and dv apart): the general kernel
        // for the next tile width, the columns past each width zero.
        if (!padded_widths_ok(p.dk, p.dv)) return LA_ERR_UNSUPPORTED;
        const bool wide = std::max(p.dk, p.dv) > 64;
        if (p.gamma) {
            if (var) return wide ? launch<128, true, true>(p) : launch<64, true, true>(p);
            return wide ? launch<128, true, false>(p) : launch<64, true, false>(p);
        }
        if (var) return wide ? launch<128, false, true>(p) : launch<64, false, true>(p);
        return wide ? launch<128, false, false>(p) : launch<64, false, false>(p);
    }
    if (p.gamma) {
        if (var) return p.dk == 128 ? launch<128, true, true>(p) : launch<64, true, true>(p);
        return p.dk == 128 ? launch<128, true, false>(p) : launch<64, true, false>(p);
    }
    // d = 64: up to 16 chunks per head, one thread-block cluster per head
    // (la_tc_causal_cluster.cu; any map and normaliser); longer sequences with enough
    // heads (elu + 1 with the normaliser), the chunk-parallel kernel
    // (la_tc_causal_chunks.cu), whose look-back needs the chunks of one head in flight
    // at a time (about twice the SM count divided by the heads) to fit its 32-chunk window.
    if (p.dk == 64 && p.N <= kClusterKernelMaxN) return causal_cluster_tc(p);
    if (var) return p.dk == 128 ? launch<128, false, true>(p) : launch<64, false, true>(p);
    if (p.dk == 64 && p.BH >= kChunkKernelMinHeads) return causal_chunks_tc(p);
    return p.dk == 128 ? launch<128, false, false>(p) : launch<64, false, false>(p);
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
