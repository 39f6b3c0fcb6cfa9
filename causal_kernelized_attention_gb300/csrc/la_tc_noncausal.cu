// Tensor-core (tcgen05 + TMA) non-causal forward, bf16 in / fp32 accumulate,
// dk = dv = D in {64, 128}.
//
// The non-causal form ("Linear attention: change the order.", mlblogg.com,
// associative trick and its NumPy implementation; "Linear Attention -- Math +
// Variants", aicassindra.com, the quadratic wall): the key-value summary of a
// head is built once, S = sum_n phi(k_n)^T v_n and z = sum_n phi(k_n), and every
// output row reads it, o_n = phi(q_n) S / max(phi(q_n) z, eps).
//
//  * One persistent CTA per SM takes work items by ticket.  Tickets first name
//    (head, split of its key chunks) items, which build the summary, then
//    (head, group of query chunks) items, which write outputs.  A CTA takes its
//    tickets in increasing order, so an output item only waits on summary items
//    whose tickets were taken before, by CTAs that are running.
//  * Summary item: per key/value chunk, S_p += phi(K_c)^T V_c and
//    z_p += phi(K_c)^T 1 in tensor memory; the split's partial (fp32) goes to
//    global memory.  The CTA that completes the last split of a head sums the
//    head's partials in split order (so the result does not depend on which CTA
//    comes last) and writes the head's state image -- the bf16 copy of S in the
//    MN-major swizzled layout of the output MMA and z as a bf16 high + low pair,
//    byte for byte as shared memory holds them -- then sets the head's ready flag.
//  * Output item: one bulk copy brings the image into shared memory (only when
//    the head changes); per query chunk O = phi(Q_c) S_bf16 and
//    qz = phi(Q_c)(z_hi + z_lo) on the tensor cores; o = O / max(qz, eps),
//    rounded to bf16 in shared memory and written by a TMA store.
//  * State mode (the prefill state of a prefix; no output items): the sums are
//    written as fp32 S and z -- by the split's own epilogue when a head has one
//    split, else by the CTA that completes the head's last split.  phi(K) is
//    evaluated in fp32 and split into bf16 high and low parts, each multiplied
//    by [V | 1] (or V and W), so the state is accurate to about 2^-17 relative
//    to fp32 phi rather than to bf16 rounding.
//
// FAVOR+ ("Linear Attention -- Math + Variants", Performer) with d = m = 64 runs
// inside this kernel (kFavor): phi(x) = exp(x W^T - |x|^2 / 2) / sqrt(m) of every Q
// and K tile replaces the tile in place.  Warp 7 issues x W^T (two N = 32 MMAs, W
// resident in shared memory) into the unused columns of the accumulators (80..111
// and 208..239, or 336..367 and 464..495: two buffers); the phi warps take
// alternate tiles, warps 8-11 the even ones and 12-15 the odd ones, one thread per
// row: the row's squared norm from shared memory, its 64 projections from TMEM,
// the exponentials written over the row.
//
// Warp roles (512 threads): warps 0-3 epilogue (TMEM lane quadrant = warp),
// warp 4 scheduler and TMA producer, warp 5 MMA issuer and TMEM owner, warp 6
// state-image loader, warp 7 idle (FAVOR+: the projection MMAs), warps 8-15 apply
// phi in shared memory.  Each
// item is published to the other roles through a small ring in shared memory.
// Every wait is bounded (mbarriers and the ready flag alike); on expiry the CTA
// records LA_ERR_TIMEOUT in this file's status word and winds down.
#include "la_common.cuh"
#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"
#include "la_tc_pad.cuh"

#include <algorithm>

namespace la {
namespace {

using namespace sm100;
using namespace tc;

static __device__ unsigned g_nc_status;

constexpr int kThreads = 512;
constexpr int kEpiThreads = 128;  // warps 0-3
constexpr int kTmaWarp = 4, kMmaWarp = 5, kImgWarp = 6, kPhiWarp0 = 8;
constexpr int kPhiThreads = 256;  // warps 8-15
constexpr int kFavorWarp = 7;     // FAVOR+: the projection MMAs
constexpr int kRing = 4;          // item ring entries
// Readers of each ring entry: 8 phi warps, the MMA thread, the loader, 4 epilogue warps.
constexpr uint32_t kRingReaders = 8 + 1 + 1 + 4;

enum : int { kEnd = 0, kSum = 1, kOut = 2 };

struct Item {
    int kind, bh, c0, nch, split;
};

// Column sums and z ride on the tensor cores in one of two ways (as in the
// causal kernel):
//  * fused (D = 64): the summary MMA's B operand is [V | 1] and the output MMA's
//    is [S_bf16 | z], one N = D + 16 MMA whose second 64-wide block (an LBO away)
//    is the ones block (column 0 = 1) or, for image slot m, the ones block's
//    columns 16(m+1) and 16(m+1)+1 holding z_hi and z_lo;
//  * separate (D = 128): N = 16 MMAs against W (summary: row 0 ones; output: the
//    image's W, rows 1 and 2 = z_hi, z_lo).
template <int D>
struct Cfg {
    static constexpr bool kFused = D == 64;
    static constexpr uint32_t kTileBytes = kC * D * 2;
    static constexpr int kStages = D == 128 ? 2 : 5;        // a stage holds K and V, or Q and the staged O
    static constexpr int kImgs = D == 128 ? 1 : 2;          // state images held at once
    static constexpr uint32_t kSbBytes = D * D * 2;
    // State image in global memory: fused = the bf16 copy of S, then z as D (hi, lo)
    // bf16 pairs; separate = W (z rows) then the bf16 copy of S.  In shared memory a
    // slot holds the S copy (fused; z goes to the ones block) or the whole image.
    static constexpr uint32_t kImgBytes = kFused ? kSbBytes + 4 * D : 2048 + kSbBytes;
    static constexpr uint32_t kSlotBytes = kFused ? kSbBytes : kImgBytes;
    // aux: fused = image slots, then the ones block (after every tile it pairs with,
    // so that LBOs are positive); separate = W (whose descriptor rows 8..15 alias into
    // the image slot after it, feeding only unread columns), then the image slot.
    static constexpr uint32_t kW = 0;
    static constexpr uint32_t kImg0 = kFused ? 0 : 2048;
    static constexpr uint32_t kOnes = kImg0 + kImgs * kSlotBytes;
    static constexpr uint32_t kAuxBytes = kFused ? kOnes + kC * 128 : kOnes;
    // Accumulator buffers in TMEM: [S or O: D columns][z or qz: 16 columns].
    static constexpr uint32_t kAccStride = D == 128 ? 256 : 128;
    static constexpr int kAcc = 512 / kAccStride;
};

template <int D>
struct alignas(1024) Smem {
    uint8_t stage[Cfg<D>::kStages][2 * Cfg<D>::kTileBytes];
    // State mode: the second buffer of low phi parts (the first is the image slots).
    // It precedes aux, so that the MMA's second 64-row block of it (16 KB on) stays
    // inside shared memory.
    uint8_t lo1[Cfg<D>::kTileBytes];
    uint8_t aux[Cfg<D>::kAuxBytes];
    uint64_t full[Cfg<D>::kStages], phi_done[Cfg<D>::kStages], empty[Cfg<D>::kStages];
    uint64_t item_full[kRing], item_empty[kRing];
    uint64_t acc_full[Cfg<D>::kAcc], acc_free[Cfg<D>::kAcc], o_staged[Cfg<D>::kAcc];
    uint64_t img_full[Cfg<D>::kImgs], img_empty[Cfg<D>::kImgs];
    uint64_t epi_sync, drain;
    uint64_t lo_free[2];  // state mode: the MMAs have read low-part buffer b
    uint64_t f_full[2], f_free[2], f_drain;  // FAVOR+: projection buffer b written / read
    Item items[kRing];
    uint32_t tmem_base;
    int abort;
    int last;      // the epilogue's CTA completed the last split of its head
    int last_cta;  // this CTA finished last: it clears the flags for the next launch
};

static_assert(sizeof(Smem<128>) <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
// State mode keeps the low phi parts of a key tile in the image slots or in lo1.
static_assert(Cfg<64>::kImgs * Cfg<64>::kSlotBytes >= Cfg<64>::kTileBytes, "no room for the low phi parts");
static_assert(Cfg<128>::kImgs * Cfg<128>::kSlotBytes >= Cfg<128>::kTileBytes, "no room for the low phi parts");
static_assert(sizeof(Smem<64>) <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

struct Params {
    float *part;         // [BH, P, D*D + D] split partials (S then z; thread-major, see add_state)
    uint8_t *img;        // [BH, kImgBytes] state images
    uint32_t *ticket;    // work ticket; ticket[1] counts finished CTAs
    uint32_t *arrived;   // [BH] completed splits per head
    uint32_t *ready;     // [BH] 1 once the head's state image is written
    int N, BH, n_chunks;
    int P, L1;           // splits per head, key chunks per split
    int T, L2;           // output items per head, query chunks per item
    float eps;
    // State mode (T = 0, no output items): the sums are written to S_out [BH, dk, dv]
    // (row = key feature) and z_out [BH, dk], fp32, row-major; null otherwise.  (Rows
    // past dk, fed by phi(0) of the zero-filled columns, are not written.)
    float *S_out, *z_out;
    // State mode, decayed state: token t of head bh weighted by gamma[bh % H]^(N-1-t)
    // (the decayed recurrence unrolled over the prefix); null otherwise.
    const float *gamma;
    int H;
    // Feature-map variant (kVar): LA_PHI_* map with shift; normalize 0: o = phi(q)^T S.
    int map;
    float shift;
    int normalize;
    // Feature widths (multiples of 8, at most D; output mode): q, k carry dk
    // columns, v, o dv; the tiles' columns past them are zero (see zero_cols).
    int dk, dv;
    // FAVOR+ (kFavor): the projection W [64, 64] bf16, row r = w_r, device memory.
    const uint16_t *favor_w;
};

// FAVOR+ projection buffers (D = 64): the columns of the accumulators past their 80
// (S or O, then z or qz), features 0..31 and 32..63 of buffer b.
__host__ __device__ constexpr uint32_t favor_lo(int b) { return b ? 336u : 80u; }
__host__ __device__ constexpr uint32_t favor_hi(int b) { return b ? 464u : 208u; }
static_assert(Cfg<64>::kAccStride == 128 && favor_lo(0) >= 64 + 16 && favor_lo(0) + 32 <= 128 &&
                  favor_hi(0) == 128 + favor_lo(0) && favor_lo(1) == 256 + favor_lo(0) && favor_hi(1) + 32 <= 512,
              "FAVOR+ projection buffers inside the accumulators' unused columns");
constexpr float kFavorLog2e = 1.4426950408889634f;

// phi of features [32 h, 32 h + 32) of row `row` of a [128 x 64] tile (128-byte
// swizzled) from their projections f: 2^((f - |x|^2 / 2) log2(e) - 3), the factor
// 1/sqrt(64) folded into the exponent; zero past the end of the sequence.
__device__ __forceinline__ void favor_half(uint8_t *tile, int row, int h, bool live, const uint32_t (&f)[32],
                                           float nrm)
{
    uint8_t *rp = tile + row * 128;
    const float cexp = fmaf(-0.5f * kFavorLog2e, nrm, -3.0f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = live ? exp2f(fmaf(__uint_as_float(f[8 * u + e]), kFavorLog2e, cexp)) : 0.f;
        *reinterpret_cast<uint4 *>(rp + (((4 * h + u) ^ (row & 7)) << 4)) =
            make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
    }
}

// State mode, decayed state or another feature map: the map (elu + 1, max(x, 0) + c
// or x + c) in fp32, times the row's weight gamma^(ebase - row) (lg = log2 gamma; 0
// without decay), split into bf16 high parts (in place) and low parts (in `lo`).
__device__ __forceinline__ float phi_map_f32(float x, int map, float c)
{
    return map == LA_PHI_RELU ? fmaxf(x, 0.f) + c : map == LA_PHI_IDENTITY ? x + c : (x > 0.f ? x + 1.f : __expf(x));
}
template <bool kVar>
__device__ __forceinline__ uint32_t phi2_split_w(uint32_t w, float wt, uint32_t *lo, int map, float c)
{
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&w);
    const float a = __bfloat162float(x.x), b = __bfloat162float(x.y);
    const float pa = (kVar ? phi_map_f32(a, map, c) : (a > 0.f ? a + 1.f : __expf(a))) * wt;
    const float pb = (kVar ? phi_map_f32(b, map, c) : (b > 0.f ? b + 1.f : __expf(b))) * wt;
    const __nv_bfloat16 ha = __float2bfloat16_rn(pa), hb = __float2bfloat16_rn(pb);
    const __nv_bfloat162 l = __floats2bfloat162_rn(pa - __bfloat162float(ha), pb - __bfloat162float(hb));
    *lo = *reinterpret_cast<const uint32_t *>(&l);
    const __nv_bfloat162 h = __halves2bfloat162(ha, hb);
    return *reinterpret_cast<const uint32_t *>(&h);
}
template <int D, int NT, bool kVar>
__device__ __forceinline__ void phi_tile_split_w(uint8_t *tile, uint8_t *lo, int t, int valid, float lg, int ebase,
                                                 int map, float c)
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
        const float wt = row < valid ? pow_decay(lg, ebase - row) : 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint4 h = make_uint4(0u, 0u, 0u, 0u), l = make_uint4(0u, 0u, 0u, 0u);
            if (row < valid) {
                h.x = phi2_split_w<kVar>(x[k].x, wt, &l.x, map, c);
                h.y = phi2_split_w<kVar>(x[k].y, wt, &l.y, map, c);
                h.z = phi2_split_w<kVar>(x[k].z, wt, &l.z, map, c);
                h.w = phi2_split_w<kVar>(x[k].w, wt, &l.w, map, c);
            }
            *reinterpret_cast<uint4 *>(tile + off + ((rot + k) & 7) * 16) = h;
            *reinterpret_cast<uint4 *>(lo + off + ((rot + k) & 7) * 16) = l;
        }
    }
}

__device__ __forceinline__ bool wait_bar(int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return tc::wait_bar(&g_nc_status, abort_flag, bar, parity);
}
__device__ __forceinline__ bool wait_bar_warp(int *abort_flag, uint64_t *bar, uint32_t parity)
{
    return tc::wait_bar_warp(&g_nc_status, abort_flag, bar, parity);
}

__device__ __forceinline__ Item decode_ticket(const Params &prm, int t)
{
    Item it{kEnd, 0, 0, 0, 0};
    const int n1 = prm.BH * prm.P, n2 = prm.BH * prm.T;
    if (t < n1) {
        it.kind = kSum;
        it.bh = t / prm.P;
        it.split = t % prm.P;
        it.c0 = it.split * prm.L1;
        it.nch = min(prm.L1, prm.n_chunks - it.c0);
    } else if (t < n1 + n2) {
        const int u = t - n1;
        it.kind = kOut;
        it.bh = u / prm.T;
        it.c0 = (u % prm.T) * prm.L2;
        it.nch = min(prm.L2, prm.n_chunks - it.c0);
    }
    return it;
}

// Sums the head's P partials (in split order) and writes its state image: the
// bf16 copy of S (MN-major, 128-byte swizzled) and z -- fused: S copy at byte 0,
// then (z_hi, z_lo) bf16 pairs; separate: W at byte 0 (row 1 = z_hi, row 2 = z_lo,
// other rows zero), then the S copy.  Run by the 128 epilogue threads; thread t
// takes state row t % D and a column range.  Two partials per round of loads.
template <int D>
__device__ __forceinline__ void build_image(const Params &prm, int bh, int t)
{
    using CF = Cfg<D>;
    constexpr int kGroups = 128 / D, kCols = D / kGroups;
    const size_t seg = (size_t)D * D + D;
    const float *part = prm.part + (size_t)bh * prm.P * seg;
    uint8_t *img = prm.img + (size_t)bh * CF::kImgBytes;
    const int i = t % D, grp = t / D;
#pragma unroll 1
    for (int cc = 0; cc < kCols; cc += 32) {
        float acc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = 0.f;
        const int col0 = grp * kCols + cc;
        int p = 0;
        for (; p + 1 < prm.P; p += 2) {
            add_state<D>(acc, part + p * seg, col0 >> 2, i);
            add_state<D>(acc, part + (p + 1) * seg, col0 >> 2, i);
        }
        if (p < prm.P) add_state<D>(acc, part + p * seg, col0 >> 2, i);
        put_sb<D>(img + (CF::kFused ? 0 : 2048), i, col0, acc);
    }
    if constexpr (CF::kFused) {
        if (t < D) {
            float zk = 0.f;
            for (int q = 0; q < prm.P; ++q) zk += __ldcg(part + q * seg + (size_t)D * D + t);
            const __nv_bfloat16 hi = __float2bfloat16_rn(zk);
            const __nv_bfloat16 lo = __float2bfloat16_rn(zk - __bfloat162float(hi));
            *reinterpret_cast<__nv_bfloat162 *>(img + CF::kSbBytes + 4 * t) = __halves2bfloat162(hi, lo);
        }
        return;
    }
    // W: thread t writes one 16-byte chunk (block t / 64, row (t / 8) % 8,
    // physical chunk t % 8, which holds logical chunk (t % 8) ^ row).
    const int blk = t >> 6, row = (t >> 3) & 7, lc = (t & 7) ^ row;
    uint32_t wv[4] = {0u, 0u, 0u, 0u};
    if (row == 1 || row == 2) {
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            float hl[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int kidx = 64 * blk + 8 * lc + e + h;
                float zk = 0.f;
                if (kidx < D)
                    for (int p = 0; p < prm.P; ++p) zk += __ldcg(part + p * seg + (size_t)D * D + kidx);
                const float hi = __bfloat162float(__float2bfloat16_rn(zk));
                hl[h] = row == 1 ? hi : zk - hi;
            }
            wv[e >> 1] = pack_bf16(hl[0], hl[1]);
        }
    }
    *reinterpret_cast<uint4 *>(img + blk * 1024 + row * 128 + (t & 7) * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
}

// State mode: sums the head's P partials in split order and writes S (fp32,
// [dk, dv] row-major, row = key feature) and z (fp32, [dk]).  Run by the 128
// epilogue threads; thread t takes row t % D and a column range.
template <int D>
__device__ __forceinline__ void write_state(const Params &prm, int bh, int t)
{
    constexpr int kGroups = 128 / D, kCols = D / kGroups;
    const size_t seg = (size_t)D * D + D;
    const float *part = prm.part + (size_t)bh * prm.P * seg;
    const int i = t % D, grp = t / D;
#pragma unroll 1
    for (int cc = 0; cc < kCols; cc += 32) {
        float acc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = 0.f;
        const int col0 = grp * kCols + cc;
        if (i >= prm.dk || col0 >= prm.dv) continue;
        int p = 0;
        for (; p + 1 < prm.P; p += 2) {
            add_state<D>(acc, part + p * seg, col0 >> 2, i);
            add_state<D>(acc, part + (p + 1) * seg, col0 >> 2, i);
        }
        if (p < prm.P) add_state<D>(acc, part + p * seg, col0 >> 2, i);
        float4 *dst = reinterpret_cast<float4 *>(prm.S_out + ((size_t)bh * prm.dk + i) * prm.dv + col0);
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
    }
    if (t < prm.dk) {
        float zk = 0.f;
        for (int q = 0; q < prm.P; ++q) zk += __ldcg(part + q * seg + (size_t)D * D + t);
        prm.z_out[(size_t)bh * prm.dk + t] = zk;
    }
}

// The epilogue threads' barrier: an mbarrier of 128 arrivals, waited on with a
// bound (a thread can arrive for the next use only after the current use has
// completed, so the phases never mix).
__device__ __forceinline__ bool epi_barrier(int *abort_flag, uint64_t *bar, uint32_t &uses)
{
    mbar_arrive(bar);
    const bool ok = wait_bar_warp(abort_flag, bar, uses & 1);
    ++uses;
    return ok;
}

template <int D, bool kVar, bool kFavor = false>
__global__ void __launch_bounds__(512, 1)
noncausal_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                    const Params prm)
{
    using CF = Cfg<D>;
    constexpr int S = CF::kStages;
    constexpr uint32_t kTile = CF::kTileBytes;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // layout assumption of the swizzled tiles
        if (threadIdx.x == 0) atomicOr(&g_nc_status, kStatusTimeout);
        return;
    }
    Smem<D> &sm = *reinterpret_cast<Smem<D> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The next launch on the stream may start its set-up now; it waits for this
    // grid to complete before it touches global memory.
    griddep_launch_dependents();

    if (tid < 128) {
        if constexpr (CF::kFused) {
            // ones block: row r holds 1 in column 0 (physical 16-byte chunk r % 8), the
            // rest zero (the z columns are written with each image)
            for (int c = tid; c < kC * 8; c += 128) {
                const uint32_t x = (c & 7) == ((c >> 3) & 7) ? 0x3F80u : 0u;
                *reinterpret_cast<uint4 *>(sm.aux + CF::kOnes + c * 16) = make_uint4(x, 0u, 0u, 0u);
            }
        } else {  // W: row 0 ones, everything else zero
            const int blk = tid >> 6, within = tid & 63;
            const uint32_t val = (within < 8) ? 0x3F803F80u : 0u;
            *reinterpret_cast<uint4 *>(sm.aux + CF::kW + blk * 1024 + within * 16) = make_uint4(val, val, val, val);
        }
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.phi_done[s], kPhiThreads);
            mbar_init(&sm.empty[s], 1);
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(&sm.item_full[r], 1);
            mbar_init(&sm.item_empty[r], kRingReaders + (kFavor ? 1 : 0));
        }
        for (int a = 0; a < CF::kAcc; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_free[a], kEpiThreads);
            mbar_init(&sm.o_staged[a], kEpiThreads);
        }
        for (int m = 0; m < CF::kImgs; ++m) {
            mbar_init(&sm.img_full[m], 1);
            mbar_init(&sm.img_empty[m], 1);
        }
        mbar_init(&sm.epi_sync, kEpiThreads);
        mbar_init(&sm.lo_free[0], 1);
        mbar_init(&sm.lo_free[1], 1);
        mbar_init(&sm.drain, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.f_full[b], 1);
            mbar_init(&sm.f_free[b], 128);
        }
        mbar_init(&sm.f_drain, 1);
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
    if constexpr (kFavor) {
        static_assert(D == 64, "FAVOR+ in the kernel: d = m = 64");
        // W into lo1 (unused outside state mode), K-major and 128-byte swizzled: the B
        // operand of x W^T, rows 0..31 for features 0..31 and rows 32..63 (4 KB on)
        if (tid < 128) {
            const uint4 *w4 = reinterpret_cast<const uint4 *>(prm.favor_w);
            for (int u = tid; u < 64 * 8; u += 128) {
                const int row = u >> 3, ch = u & 7;
                *reinterpret_cast<uint4 *>(sm.lo1 + row * 128 + ((ch ^ (row & 7)) << 4)) = __ldg(w4 + u);
            }
            fence_proxy_async_smem();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    int *abort_flag = &sm.abort;

    if (warp >= kPhiWarp0) {
        // ---------------------------------------------------------------- phi warps
        const int t = tid - kPhiWarp0 * 32;
        int j = 0;
        for (int it = 0;; ++it) {
            const int r = it % kRing;
            if (!wait_bar_warp(abort_flag, &sm.item_full[r], (it / kRing) & 1)) break;
            const Item item = sm.items[r];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.item_empty[r]);
            if (item.kind == kEnd) break;
            bool ok = true;
            for (int c = 0; c < item.nch; ++c, ++j) {
                const int s = j % S;
                if (!(ok = wait_bar_warp(abort_flag, &sm.full[s], (j / S) & 1))) break;
                // K (summary) or Q (output) is the first tile of the stage.
                const int valid = prm.N - (item.c0 + c) * kC;
                if (prm.S_out) {
                    // State mode: phi in fp32, split into bf16 high parts (in place) and
                    // low parts (buffer j % 2: the unused image slots or lo1), once the
                    // MMAs of the tile two before have read that buffer.
                    const int b = j & 1, n = j >> 1;
                    if (n > 0 && !(ok = wait_bar_warp(abort_flag, &sm.lo_free[b], (n - 1) & 1))) break;
                    if (kVar || prm.gamma)
                        phi_tile_split_w<D, kPhiThreads, kVar>(sm.stage[s], b ? sm.lo1 : sm.aux + CF::kImg0, t, valid,
                                                         prm.gamma ? log2f(__ldg(prm.gamma + item.bh % prm.H)) : 0.f,
                                                         prm.N - 1 - (item.c0 + c) * kC, prm.map, prm.shift);
                    else
                        phi_tile_split<D, kPhiThreads>(sm.stage[s], b ? sm.lo1 : sm.aux + CF::kImg0, t, valid);
                } else if constexpr (kFavor) {
                    // tile j: warps 8-11 if j is even, 12-15 if odd; buffer j % 2
                    const int b = j & 1, n = j >> 1;
                    if (((warp - kPhiWarp0) >> 2) == b) {
                        const int row = 32 * (warp & 3) + lane;
                        const uint8_t *rp = sm.stage[s] + row * 128;
                        float nrm = 0.f;
#pragma unroll
                        for (int u = 0; u < 8; ++u) {  // any chunk order covers the row
                            const uint4 w4 = *reinterpret_cast<const uint4 *>(rp + (((u + row) & 7) << 4));
                            const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv[e]));
                                nrm = fmaf(f.x, f.x, nrm);
                                nrm = fmaf(f.y, f.y, nrm);
                            }
                        }
                        if (!(ok = wait_bar_warp(abort_flag, &sm.f_full[b], n & 1))) break;
                        tc_fence_after();
                        const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll 1
                        for (int h = 0; h < 2; ++h) {
                            uint32_t f[32];
                            tmem_ld32(tq + (h ? favor_hi(b) : favor_lo(b)), f);
                            tmem_ld_wait();
                            favor_half(sm.stage[s], row, h, row < valid, f, nrm);
                        }
                        tc_fence_before();
                        mbar_arrive(&sm.f_free[b]);  // both halves read from TMEM
                    }
                } else {
                    phi_tile<D, kPhiThreads, false, kVar>(sm.stage[s], t, valid, 0.f, 0, prm.map, prm.shift);
                    if (prm.dk < D && item.kind == kSum) zero_cols<D>(sm.stage[s], t, kPhiThreads, prm.dk);
                }
                fence_proxy_async_smem();
                mbar_arrive(&sm.phi_done[s]);
            }
            if (!ok) break;
        }
    } else if (warp == kTmaWarp) {
        // ---------------------------------------------------------------- scheduler + TMA producer
        if (lane == 0) {
            tma_prefetch_map(&map_q);
            tma_prefetch_map(&map_k);
            tma_prefetch_map(&map_v);
            tma_prefetch_map(&map_o);
            // Every tile is read once: let it leave L2 first, ahead of the partials and
            // state images that other CTAs read back.
            const uint64_t pol_once = l2_policy_evict_first();
            int j = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int r = it % kRing;
                if (it >= kRing && !(ok = wait_bar(abort_flag, &sm.item_empty[r], ((it / kRing) - 1) & 1))) break;
                const Item item = decode_ticket(prm, (int)atomicAdd(prm.ticket, 1u));
                sm.items[r] = item;
                mbar_arrive(&sm.item_full[r]);
                if (item.kind == kEnd) break;
                for (int c = 0; c < item.nch; ++c, ++j) {
                    const int s = j % S, rr = j / S;
                    if (rr > 0 && !(ok = wait_bar(abort_flag, &sm.empty[s], (rr - 1) & 1))) break;
                    const int row0 = (item.c0 + c) * kC;
                    uint8_t *st = sm.stage[s];
                    if (item.kind == kSum) {
                        mbar_arrive_expect_tx(&sm.full[s], 2 * kTile);
#pragma unroll
                        for (int b = 0; b < D / 64; ++b) {
                            tma_load_3d_hint(st + b * kBox, &map_k, &sm.full[s], 64 * b, row0, item.bh, pol_once);
                            tma_load_3d_hint(st + kTile + b * kBox, &map_v, &sm.full[s], 64 * b, row0, item.bh, pol_once);
                        }
                    } else {
                        mbar_arrive_expect_tx(&sm.full[s], kTile);
#pragma unroll
                        for (int b = 0; b < D / 64; ++b)
                            tma_load_3d_hint(st + b * kBox, &map_q, &sm.full[s], 64 * b, row0, item.bh, pol_once);
                    }
                }
            }
            // No copy may still be writing shared memory when the CTA exits.
            for (int jj = max(0, j - S); jj < j; ++jj) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&sm.full[jj % S], (jj / S) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr int NE = CF::kFused ? D + 16 : D;  // N of the MMAs against V or S
            const uint32_t id_KV = idesc_bf16_f32(128, NE, true, true);   // phi(K)^T [V | 1]
            const uint32_t id_KW = idesc_bf16_f32(128, 16, true, false);  // phi(K)^T W^T
            const uint32_t id_QS = idesc_bf16_f32(128, NE, false, true);  // phi(Q) [S_bf16 | z]
            const uint32_t id_QW = idesc_bf16_f32(128, 16, false, false); // phi(Q) W^T
            const uint32_t aux = smem_u32(sm.aux);
            const uint32_t w1 = aux + CF::kW, ones = aux + CF::kOnes;
            int j = 0, q = 0, n_img = 0, cur_bh = -1, cur_m = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int r = it % kRing;
                if (!(ok = wait_bar(abort_flag, &sm.item_full[r], (it / kRing) & 1))) break;
                const Item item = sm.items[r];
                mbar_arrive(&sm.item_empty[r]);
                if (item.kind == kEnd) break;
                if (item.kind == kSum) {
                    const int a = q % CF::kAcc;
                    if (q >= CF::kAcc && !(ok = wait_bar(abort_flag, &sm.acc_free[a], ((q / CF::kAcc) - 1) & 1)))
                        break;
                    tc_fence_after();
                    const uint32_t dS = tmem + a * CF::kAccStride, dZ = dS + D;
                    for (int c = 0; c < item.nch; ++c, ++j) {
                        const int s = j % S;
                        if (!(ok = wait_bar(abort_flag, &sm.phi_done[s], (j / S) & 1))) break;
                        tc_fence_after();
                        // phi(K)^T is MN-major with its second 64-row block one box on
                        // (for D = 64 that is the V tile: rows 64..127 are never read).
                        const uint32_t ka = smem_u32(sm.stage[s]), va = ka + kTile;
                        const uint32_t lbo_v = CF::kFused ? ones - va : kBox;  // [V | 1] or V's second box
#pragma unroll
                        for (int kk = 0; kk < kC / 16; ++kk) {
                            const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
                            mma_ss(dS, mnmajor(ka, kk, kBox), mnmajor(va, kk, lbo_v), id_KV, acc);
                            if constexpr (!CF::kFused)
                                mma_ss(dZ, mnmajor(ka, kk, kBox), wdesc(w1, kk), id_KW, acc);
                        }
                        if (prm.S_out) {  // state mode: the low phi parts against the same V (and 1)
                            const uint32_t la = (j & 1) ? smem_u32(sm.lo1) : aux + CF::kImg0;
#pragma unroll
                            for (int kk = 0; kk < kC / 16; ++kk) {
                                mma_ss(dS, mnmajor(la, kk, kBox), mnmajor(va, kk, lbo_v), id_KV, 1u);
                                if constexpr (!CF::kFused)
                                    mma_ss(dZ, mnmajor(la, kk, kBox), wdesc(w1, kk), id_KW, 1u);
                            }
                            mma_commit(&sm.lo_free[j & 1]);
                        }
                        mma_commit(&sm.empty[s]);
                    }
                    if (!ok) break;
                    mma_commit(&sm.acc_full[a]);
                    ++q;
                } else {
                    if (item.bh != cur_bh) {  // next state image; the one before it is free once
                        const int m = n_img % CF::kImgs;  // every MMA issued so far completes
                        if (n_img > 0) mma_commit(&sm.img_empty[(n_img - 1) % CF::kImgs]);
                        if (!(ok = wait_bar(abort_flag, &sm.img_full[m], (n_img / CF::kImgs) & 1))) break;
                        cur_bh = item.bh;
                        cur_m = m;
                        ++n_img;
                    }
                    // separate: W then the S copy in the slot; fused: the S copy, its z in
                    // the ones block's columns 16(m+1), 16(m+1)+1 (32(m+1) bytes on)
                    const uint32_t slot = aux + CF::kImg0 + cur_m * CF::kSlotBytes;
                    const uint32_t w2 = slot, sb = CF::kFused ? slot : slot + 2048;
                    const uint32_t lbo_sb = CF::kFused ? ones + 32 * (cur_m + 1) - sb : D * 128;
                    for (int c = 0; c < item.nch; ++c, ++j, ++q) {
                        const int s = j % S, a = q % CF::kAcc;
                        if (!(ok = wait_bar(abort_flag, &sm.phi_done[s], (j / S) & 1))) break;
                        if (q >= CF::kAcc && !(ok = wait_bar(abort_flag, &sm.acc_free[a], ((q / CF::kAcc) - 1) & 1)))
                            break;
                        tc_fence_after();
                        const uint32_t qa = smem_u32(sm.stage[s]);
                        const uint32_t dO = tmem + a * CF::kAccStride, dQZ = dO + D;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            mma_ss(dO, kmajor(qa, kk), mnmajor(sb, kk, lbo_sb), id_QS, kk > 0 ? 1u : 0u);
                            if constexpr (!CF::kFused)
                                mma_ss(dQZ, kmajor(qa, kk), wdesc(w2, kk), id_QW, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&sm.acc_full[a]);
                    }
                }
            }
            // all issued MMAs complete before TMEM is freed
            mma_commit(&sm.drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&sm.drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else if (kFavor && warp == kFavorWarp) {
        // ---------------------------------------------------------------- FAVOR+ projections
        if (lane == 0) {
            const uint32_t wa = smem_u32(sm.lo1);
            const uint32_t id = idesc_bf16_f32(128, 32, false, false);  // x W^T, 32 features a group
            int j = 0;
            bool ok = true, issued = false;
            for (int it = 0; ok; ++it) {
                const int r = it % kRing;
                if (!(ok = wait_bar(abort_flag, &sm.item_full[r], (it / kRing) & 1))) break;
                const Item item = sm.items[r];
                mbar_arrive(&sm.item_empty[r]);
                if (item.kind == kEnd) break;
                for (int c = 0; c < item.nch; ++c, ++j) {
                    const int s = j % S, b = j & 1, n = j >> 1;
                    if (!(ok = wait_bar(abort_flag, &sm.full[s], (j / S) & 1))) break;
                    if (n > 0 && !(ok = wait_bar(abort_flag, &sm.f_free[b], (n - 1) & 1))) break;
                    tc_fence_after();
                    const uint32_t xa = smem_u32(sm.stage[s]);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + favor_lo(b), kmajor(xa, kk), kmajor(wa, kk), id, kk > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + favor_hi(b), kmajor(xa, kk), kmajor(wa + 32 * 128, kk), id, kk > 0 ? 1u : 0u);
                    mma_commit(&sm.f_full[b]);
                    issued = true;
                }
            }
            if (issued) {  // every projection issued completes before TMEM is freed
                mma_commit(&sm.f_drain);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&sm.f_drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == kImgWarp) {
        // ---------------------------------------------------------------- state-image loader
        if (lane == 0) {
            int n_img = 0, cur_bh = -1;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int r = it % kRing;
                if (!(ok = wait_bar(abort_flag, &sm.item_full[r], (it / kRing) & 1))) break;
                const Item item = sm.items[r];
                mbar_arrive(&sm.item_empty[r]);
                if (item.kind == kEnd) break;
                if (item.kind != kOut || item.bh == cur_bh) continue;
                const int m = n_img % CF::kImgs;
                if (n_img >= CF::kImgs && !(ok = wait_bar(abort_flag, &sm.img_empty[m], ((n_img / CF::kImgs) - 1) & 1)))
                    break;
                // The head's summary is complete once its ready flag is set (bounded wait).
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_gpu(prm.ready + item.bh) == 0u) {
                    if (aborted(abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (globaltimer_ns() - t0 > kWaitLimitNs) {
                        *(volatile int *)abort_flag = 1;
                        atomicOr(&g_nc_status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    __nanosleep(256);
                }
                if (!ok) break;
                fence_proxy_async_global();
                const uint8_t *src = prm.img + (size_t)item.bh * CF::kImgBytes;
                uint8_t *slot = sm.aux + CF::kImg0 + m * CF::kSlotBytes;
                if constexpr (CF::kFused) {
                    // z (hi, lo) pairs into the ones block's columns 16(m+1), 16(m+1)+1
                    const uint4 *zs = reinterpret_cast<const uint4 *>(src + CF::kSbBytes);
                    for (int x = 0; x < D / 4; ++x) {
                        const uint4 z4 = __ldcg(zs + x);
                        const uint32_t zz[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<uint32_t *>(sm.aux + CF::kOnes + sw128_offset(4 * x + e, 16 * (m + 1))) =
                                zz[e];
                    }
                    fence_proxy_async_smem();
                }
                mbar_arrive_expect_tx(&sm.img_full[m], CF::kSlotBytes);
                bulk_load(slot, src, CF::kSlotBytes, &sm.img_full[m]);
                cur_bh = item.bh;
                ++n_img;
            }
            // No copy may still be writing shared memory when the CTA exits.
            for (int n = max(0, n_img - CF::kImgs); n < n_img; ++n) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&sm.img_full[n % CF::kImgs], (n / CF::kImgs) & 1) &&
                       globaltimer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp < kEpiThreads / 32) {
        // ---------------------------------------------------------------- epilogue warps 0-3
        const int i = tid;  // TMEM lane = state row (summary) or query row (output)
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        const bool leader = tid == 0;
        const size_t seg = (size_t)D * D + D;
        int j = 0, q = 0, prev_stage = -1;
        uint32_t syncs = 0;
        // Phase bit of each o_staged[a]: those barriers advance only on output
        // jobs, while q also counts summary jobs.
        uint32_t ostaged_phase = 0;
        for (int it = 0;; ++it) {
            const int r = it % kRing;
            if (!wait_bar_warp(abort_flag, &sm.item_full[r], (it / kRing) & 1)) break;
            const Item item = sm.items[r];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.item_empty[r]);
            if (item.kind == kEnd) break;
            if (item.kind == kSum) {
                const int a = q % CF::kAcc;
                if (!wait_bar_warp(abort_flag, &sm.acc_full[a], (q / CF::kAcc) & 1)) break;
                tc_fence_after();
                const uint32_t ta = tl + a * CF::kAccStride;
                // State mode with one split per head: the sums go straight to S_out, z_out.
                const bool state_now = prm.S_out != nullptr && prm.P == 1;
                float *dst = prm.part + ((size_t)item.bh * prm.P + item.split) * seg;
#pragma unroll 1
                for (int cc = 0; cc < D; cc += 32) {
                    uint32_t v[32];
                    tmem_ld32(ta + cc, v);
                    tmem_ld_wait();
                    if (i < D && state_now) {
                        if (i >= prm.dk || cc >= prm.dv) continue;  // (after the warp-wide tmem_ld32)
                        float4 *d4 = reinterpret_cast<float4 *>(prm.S_out + ((size_t)item.bh * prm.dk + i) * prm.dv + cc);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            d4[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                    } else if (i < D) {
                        float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            d4[(size_t)((cc >> 2) + e) * D + i] =
                                make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                            __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                    }
                }
                const float zs = __uint_as_float(tmem_ld1(ta + D));
                tmem_ld_wait();
                if (i < D) {
                    if (state_now) {
                        if (i < prm.dk) prm.z_out[(size_t)item.bh * prm.dk + i] = zs;
                    } else
                        dst[(size_t)D * D + i] = zs;
                }
                tc_fence_before();
                mbar_arrive(&sm.acc_free[a]);
                ++q;
                j += item.nch;
                if (state_now) continue;
                // Count the split; the CTA that completes the head's last split builds its
                // image.  The barrier (mbarrier arrive/wait: release/acquire at CTA scope)
                // orders every thread's partial writes before the leader's acq_rel atomic,
                // whose release is cumulative: no fence per thread is needed.
                if (!epi_barrier(abort_flag, &sm.epi_sync, syncs)) break;
                if (leader) sm.last = atom_add_acq_rel_gpu(prm.arrived + item.bh, 1u) == (uint32_t)(prm.P - 1);
                if (!epi_barrier(abort_flag, &sm.epi_sync, syncs)) break;
                if (sm.last && prm.S_out) {  // state mode: the sums are the result
                    fence_acq_rel_gpu();
                    write_state<D>(prm, item.bh, tid);
                } else if (sm.last) {
                    fence_acq_rel_gpu();
                    build_image<D>(prm, item.bh, tid);
                    fence_acq_rel_gpu();
                    fence_proxy_async_global();
                    if (!epi_barrier(abort_flag, &sm.epi_sync, syncs)) break;
                    if (leader) st_release_gpu(prm.ready + item.bh, 1u);
                }
            } else {
                bool ok = true;
                for (int c = 0; c < item.nch; ++c, ++j, ++q) {
                    const int s = j % S, a = q % CF::kAcc;
                    if (!(ok = wait_bar_warp(abort_flag, &sm.acc_full[a], (q / CF::kAcc) & 1))) break;
                    tc_fence_after();
                    const uint32_t ta = tl + a * CF::kAccStride;
                    float inv;
                    {
                        // phi(q) z_hi and phi(q) z_lo: fused in columns D, D + 1; separate
                        // in columns D + 1, D + 2 (W rows 1 and 2)
                        uint32_t qz[32];
                        if constexpr (kFavor)  // columns 80.. hold projections being written
                            tmem_ld16(ta + D, *reinterpret_cast<uint32_t(*)[16]>(&qz[0]));
                        else
                            tmem_ld32(ta + D, qz);
                        tmem_ld_wait();
                        constexpr int zc = CF::kFused ? 0 : 1;
                        inv = (kVar && !prm.normalize)
                                  ? 1.f
                                  : 1.f / fmaxf(__uint_as_float(qz[zc]) + __uint_as_float(qz[zc + 1]), prm.eps);
                    }
                    uint8_t *ost = sm.stage[s] + kTile;  // the second tile of the stage stages O
#pragma unroll 1
                    for (int cc = 0; cc < D / 64 && 64 * cc < prm.dv; ++cc) {  // (columns past dv are not stored)
                        uint32_t v[64];
                        tmem_ld32(ta + cc * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                        tmem_ld32(ta + cc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                        tmem_ld_wait();
                        uint8_t *rowp = ost + cc * kBox + i * 128;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            *reinterpret_cast<uint4 *>(rowp + ((u ^ (i & 7)) << 4)) = make_uint4(
                                pack_bf16(__uint_as_float(v[8 * u]) * inv, __uint_as_float(v[8 * u + 1]) * inv),
                                pack_bf16(__uint_as_float(v[8 * u + 2]) * inv, __uint_as_float(v[8 * u + 3]) * inv),
                                pack_bf16(__uint_as_float(v[8 * u + 4]) * inv, __uint_as_float(v[8 * u + 5]) * inv),
                                pack_bf16(__uint_as_float(v[8 * u + 6]) * inv, __uint_as_float(v[8 * u + 7]) * inv));
                    }
                    // o_staged before acc_free: buffer a is refilled only after every
                    // thread has arrived on acc_free[a], hence on o_staged[a] as well.
                    fence_proxy_async_smem();
                    mbar_arrive(&sm.o_staged[a]);
                    tc_fence_before();
                    mbar_arrive(&sm.acc_free[a]);
                    if (leader && (ok = wait_bar(abort_flag, &sm.o_staged[a], (ostaged_phase >> a) & 1u))) {
                        const uint64_t pol_once = l2_policy_evict_first();
#pragma unroll
                        for (int cc = 0; cc < D / 64; ++cc)
                            if (64 * cc < prm.dv)
                                tma_store_3d_hint(&map_o, ost + cc * kBox, 64 * cc, (item.c0 + c) * kC, item.bh, pol_once);
                        tma_store_commit();
                        // The previous tile's store has read its staged O: that stage may be refilled.
                        tma_store_wait_read<1>();
                        if (prev_stage >= 0) mbar_arrive(&sm.empty[prev_stage]);
                        prev_stage = s;
                    }
                    ostaged_phase ^= 1u << a;
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;  // the whole warp leaves together
                }
                if (!ok) break;
            }
        }
        if (leader) {
            tma_store_wait_read_all();
            if (prev_stage >= 0) mbar_arrive(&sm.empty[prev_stage]);
            tma_store_wait_all();  // all output stores complete before the CTA exits
        }
    }

    tc_fence_before();
    __threadfence();  // this CTA's flag traffic is done before it counts itself finished
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
    // The last CTA to finish leaves the ticket, the counter and the per-head flags
    // at zero, ready for the next launch on the same flags.
    if (tid == 0) sm.last_cta = atom_add_acq_rel_gpu(prm.ticket + 1, 1u) == gridDim.x - 1;
    __syncthreads();
    if (sm.last_cta) {
        for (int x = tid; x < 2 * prm.BH; x += kThreads) prm.arrived[x] = 0u;  // arrived then ready
        if (tid == 0) {
            prm.ticket[0] = 0u;
            prm.ticket[1] = 0u;
        }
    }
}

// ------------------------------------------------------------------ host side
template <int D, bool kVar, bool kFavor = false>
la_status launch(const Problem &p, float *S_out = nullptr, float *z_out = nullptr, const void *favor_w = nullptr)
{
    using CF = Cfg<D>;
    // State mode (S_out given): summary items only; the q and o maps are never used
    // and are built on k.
    const bool state = S_out != nullptr;
    CUtensorMap mq, mk, mv, mo;
    la_status st = make_map(&mq, state ? p.k : p.q, p.BH, p.N, p.dk);
    if (st == LA_OK) st = make_map(&mk, p.k, p.BH, p.N, p.dk);
    if (st == LA_OK) st = make_map(&mv, p.v, p.BH, p.N, p.dv);
    if (st == LA_OK) st = make_map(&mo, state ? p.k : p.o, p.BH, p.N, state ? p.dk : p.dv);
    if (st != LA_OK) return st;

    const int n_chunks = ceil_div(p.N, kC);
    const int n_sm = sm_count();
    // About two summary items and four output items per SM: enough to balance
    // the persistent CTAs; at most 32 partials per head for its last CTA to sum.
    int P = std::min(std::min(32, n_chunks), std::max(1, ceil_div(2 * n_sm, p.BH)));
    const int L1 = ceil_div(n_chunks, P);
    P = ceil_div(n_chunks, L1);
    int T = 0, L2 = 1;
    if (!state) {
        T = std::min(n_chunks, std::max(1, ceil_div(4 * n_sm, p.BH)));
        L2 = ceil_div(n_chunks, T);
        T = ceil_div(n_chunks, L2);
    }
    const long long items = (long long)p.BH * (P + T);
    if (items > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;

    const size_t seg = (size_t)D * D + D;
    const size_t flag_bytes = ((16 + (size_t)p.BH * 8) + 255) / 256 * 256;
    // (state mode with one split per head writes the sums directly: no partials)
    const size_t part_bytes = state && P == 1 ? 0 : ((size_t)p.BH * P * seg * 4 + 255) / 256 * 256;
    const size_t img_bytes = state ? 0 : (size_t)p.BH * CF::kImgBytes;

    // Flags, partials and images from the stream's workspaces (flags already zero)
    // when they can serve the call, else from per-call scratch (flags cleared by a
    // memset).  With both workspaces, consecutive calls on the stream are kernel
    // after kernel, which lets a launch overlap the tail of the one before it.
    void *ws = nullptr, *data = nullptr;
    st = flag_workspace(p.stream, flag_bytes, &ws);
    if (st != LA_OK && st != LA_ERR_UNSUPPORTED) return st;
    st = data_workspace(p.stream, part_bytes + img_bytes, &data);
    if (st != LA_OK && st != LA_ERR_UNSUPPORTED) return st;
    const size_t own_flags = ws ? 0 : flag_bytes;
    const size_t own_data = data ? 0 : part_bytes + img_bytes;
    Scratch scratch;
    if (own_flags + own_data > 0) {
        st = scratch.alloc(own_flags + own_data, p.stream);
        if (st != LA_OK) return st;
    }
    uint8_t *base = (uint8_t *)scratch.ptr;
    uint8_t *flags = ws ? (uint8_t *)ws : base;
    uint8_t *work = data ? (uint8_t *)data : base + own_flags;
    if (!ws) {
        cudaError_t e = cudaMemsetAsync(flags, 0, flag_bytes, p.stream);
        count_launches();
        if (e != cudaSuccess) return cuda_status(e);
    }

    Params prm;
    prm.ticket = (uint32_t *)flags;
    prm.arrived = (uint32_t *)(flags + 16);
    prm.ready = prm.arrived + p.BH;
    prm.part = (float *)work;
    prm.img = work + part_bytes;
    prm.N = p.N;
    prm.BH = p.BH;
    prm.n_chunks = n_chunks;
    prm.P = P;
    prm.L1 = L1;
    prm.T = T;
    prm.L2 = L2;
    prm.eps = p.eps;
    prm.S_out = S_out;
    prm.z_out = z_out;
    prm.gamma = state ? p.gamma : nullptr;
    prm.H = p.H;
    prm.map = p.var.map;
    prm.shift = p.var.shift;
    prm.normalize = p.var.normalize;
    prm.dk = p.dk;
    prm.dv = p.dv;
    prm.favor_w = (const uint16_t *)favor_w;

    const int smem = (int)sizeof(Smem<D>);
    auto kern = noncausal_tc_kernel<D, kVar, kFavor>;
    st = ensure_smem((const void *)kern, smem);
    if (st != LA_OK) return st;
    const unsigned grid = (unsigned)std::min<long long>(items, n_sm);
    count_launches();
    return launch_dependent(kern, grid, kThreads, smem, p.stream, mq, mk, mv, mo, prm);
}

}  // namespace

la_status noncausal_tc(const Problem &p)
{
    if (p.dtype != LA_BF16 || p.N < kC || !padded_widths_ok(p.dk, p.dv)) return LA_ERR_UNSUPPORTED;
    // dk = dv = 64 or 128, or other widths on the next tile width (columns past each
    // width zero)
    const bool wide = std::max(p.dk, p.dv) > 64;
    if (!p.var.is_default()) return wide ? launch<128, true>(p) : launch<64, true>(p);
    return wide ? launch<128, false>(p) : launch<64, false>(p);
}

la_status noncausal_tc_favor(const Problem &p, const void *w)
{
    // FAVOR+ features in the kernel: d = m = 64 (the features replace the tiles in
    // place), dv up to 64, the identity map on the features with the normaliser.
    if (p.dtype != LA_BF16 || p.N < kC || p.dk != 64 || p.dv > 64 || !padded_widths_ok(p.dk, p.dv) || !w ||
        ((uintptr_t)w & 15u) != 0)
        return LA_ERR_UNSUPPORTED;
    Problem q = p;
    q.var = Variant();
    return launch<64, false, true>(q, nullptr, nullptr, w);
}

la_status noncausal_tc_state(const void *k, const void *v, float *S, float *z, int BH, int N, int dk, int dv,
                             cudaStream_t stream, const float *gamma, int H, const Variant &var)
{
    if (N < kC || !padded_widths_ok(dk, dv)) return LA_ERR_UNSUPPORTED;
    const int D = std::max(dk, dv) > 64 ? 128 : 64;
    Problem p{};
    p.q = k;
    p.k = k;
    p.v = v;
    p.o = nullptr;
    p.BH = BH;
    p.N = N;
    p.dk = dk;
    p.dv = dv;
    p.chunk = kC;
    p.eps = 0.f;
    p.dtype = LA_BF16;
    p.stream = stream;
    p.gamma = gamma;
    p.H = H;
    // the state does not depend on the normaliser: only a map other than elu + 1 is a variant
    p.var.map = var.map;
    p.var.shift = var.shift;
    if (var.map != LA_PHI_ELU1) return D == 128 ? launch<128, true>(p, S, z) : launch<64, true>(p, S, z);
    return D == 128 ? launch<128, false>(p, S, z) : launch<64, false>(p, S, z);
}

la_status tc_noncausal_read_status(cudaStream_t s, unsigned *bits)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_nc_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_nc_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // namespace la
