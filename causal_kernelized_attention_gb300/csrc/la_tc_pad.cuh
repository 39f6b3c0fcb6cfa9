// Feature widths below the tile width on the tensor-core forward kernels.
//
// A kernel built for D columns (64 or 128) serves dk, dv <= D (multiples of 8):
// the tensor maps carry the true widths, so TMA fills the columns past them
// with zeros and clips them from the stores.  phi maps those zeros to phi(0),
// which is 1 for elu + 1 (and the shift for the variants): in phi(K) that
// would add a phantom feature to every score and to z.  zero_cols rewrites them
// to 0 in phi(K) only; phi(Q)'s extra columns then meet zero rows of S, zero
// entries of z and zero columns of phi(K) in every product, so they drop out.
#pragma once

#include <cstdint>

#include "la_tc_common.cuh"

namespace la {
namespace tc {

// Zeroes columns >= live of a phi'd [128 x D] tile (D / 64 boxes of 128-byte
// swizzled rows), over the unit partition of phi_tile and phi_tile_rolled (unit
// u: row u % 128, half (u / 128) % 2 of box u / 256, units t, t + nt, ...), so a
// thread rewrites only chunks it wrote itself and needs no barrier after phi.
// Widths the padded tiles serve: whole 16-byte rows for TMA, within 128 columns.
inline bool padded_widths_ok(int dk, int dv)
{
    return dk >= 8 && dv >= 8 && dk <= 128 && dv <= 128 && dk % 8 == 0 && dv % 8 == 0;
}

template <int D>
__device__ __forceinline__ void zero_cols(uint8_t *tile, int t, int nt, int live)
{
    constexpr int kUnits = 128 * (D / 32);
#pragma unroll 1
    for (int u = t; u < kUnits; u += nt) {
        const int row = u & 127, hb = u >> 7, box = hb >> 1;
        uint8_t *rp = tile + box * kBox + row * 128;
        const int rot = row + (hb & 1) * 4;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int phys = (rot + k) & 7;              // the chunk phi rewrote
            const int col = 64 * box + 8 * (phys ^ (row & 7));  // its first logical column
            if (col >= live) *reinterpret_cast<uint4 *>(rp + phys * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

}  // namespace tc
}  // namespace la
