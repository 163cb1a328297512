// Residue-class tensor maps: operands of any alignment read in place by the
// TMA (shared by the FFMA and the three-product TF32 kernels).
//
// A tensor map needs a 16-byte aligned base and a row pitch that is a
// multiple of 16 bytes.  Rows r = 4q + j of one residue class j (mod 4) lie
// 4 ld floats = 16 ld bytes apart, a multiple of 16, so every row of a class
// starts at the same offset t_j (0..3 floats) inside its 16-byte block: one
// map per class, based at the block boundary before row j, addresses them
// all.  Each pipeline stage loads, per class, a box starting at the block
// boundary that covers the slice's elements wherever t_j puts them (32 k + 3
// of A, 128 columns + 3 of B: boxes of 36 and 132 floats, no swizzle): A's
// element (m, k) of the slice sits in class m mod 4's box, row m / 4, at
// t_{m mod 4} + k; B's element (k, n) in class k mod 4's box, row k / 4, at
// t_{k mod 4} + n.  Elements left of a row's start (the previous row's tail,
// inside the same 16-byte block) land in the box but are never read; each
// map's extent ends at its rows' last element, so everything past it reads
// as the tensor map's zero fill.  The host encodes the maps (encode_res) and
// passes the offsets t_j two bits each (bits 2j, 2j + 1).
#pragma once

#include <cuda.h>

namespace gb300 {

constexpr int kResTileRows = 128;  // rows of A per tile (32 per class)
constexpr int kResTileCols = 128;  // columns of B per tile
constexpr int kResSliceK = 32;     // k per slice (8 rows of B per class)
constexpr int kResABox = kResSliceK + 4;                            // floats per A box row
constexpr int kResBBox = kResTileCols + 4;                          // floats per B box row
constexpr int kResAPlaneBytes = (kResTileRows / 4) * kResABox * 4;  // one class of an A slice (4608 B)
constexpr int kResBPlaneBytes = (kResSliceK / 4) * kResBBox * 4;    // one class of a B slice (4224 B)
static_assert(kResAPlaneBytes % 128 == 0 && kResBPlaneBytes % 128 == 0, "tensor-copy destinations: 128-byte aligned");

struct ResMaps {
    CUtensorMap m[4];  // residue classes j = 0..3
};
// The kernel parameter type of an operand's maps: four class maps, or one.
template <bool RES>
struct MapsForT {
    using type = CUtensorMap;
};
template <>
struct MapsForT<true> {
    using type = ResMaps;
};
template <bool RES>
using MapsFor = typename MapsForT<RES>::type;

#ifdef __CUDACC__
__device__ __forceinline__ const CUtensorMap& res_map(const ResMaps& r, int j) { return r.m[j]; }
__device__ __forceinline__ const CUtensorMap& res_map(const CUtensorMap& r, int) { return r; }
// t_j of a packed shift word.
__device__ __forceinline__ int res_shift(int packed, int j) { return (packed >> (2 * j)) & 3; }
#endif

}  // namespace gb300
