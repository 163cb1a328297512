// Tile shape, shared-memory budget, instruction descriptor and kernel
// parameters of the three-product TF32 tensor-core kernel (host and device).
#pragma once

#include <cstdint>

#include "res_maps.cuh"

namespace gb300 {

constexpr int kTcBM = 128;
constexpr int kTcBN = 128;
constexpr int kTcBK = 32;
constexpr int kTcSplitWarps = 8;                // warps that split K-slices into TF32 parts
constexpr int kTcThreads = 64 + 32 * kTcSplitWarps;
constexpr int kTcRawABytes = kTcBM * kTcBK * 4;  // 16 KiB: TMA A slice, 128-byte swizzled rows
constexpr int kTcRawBBytes = kTcBK * kTcBN * 4;  // 16 KiB: TMA B slice, 512-byte rows
constexpr int kTcOpBytes = 128 * kTcBK * 4;      // 16 KiB: one K-major operand tile
constexpr int kTcSplitBytes = 4 * kTcOpBytes;    // A_big, A_small, B_big, B_small
constexpr int kTcRawStages = 3;
constexpr int kTcSplitStages = 2;
constexpr int kTcTmemCols = 128;
constexpr unsigned kTcStatusTimeout = 4u;
constexpr int kTcRingBytes = kTcRawStages * (kTcRawABytes + kTcRawBBytes) + kTcSplitStages * kTcSplitBytes;
constexpr int kTcSmemBytes = kTcRingBytes + 1024 /*align*/ + 256 /*barriers*/;

// Instruction descriptor of tcgen05.mma.kind::tf32: D FP32 (bits 4-5 = 1),
// A and B TF32 (bits 7-9 = bits 10-12 = 2), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kTcIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(kTcBN >> 3) << 17) |
                              (static_cast<uint32_t>(kTcBM >> 4) << 24);

// Shapes of the split-tile kernel, sgemm_3xtf32_kernel<BN, BK>: 128 x BN
// output tiles, K-slices of BK.  <128, 32> (variant 1): 128-byte operand rows
// (128-byte swizzle), 3 raw and 2 split stages, 224 KiB.  <256, 16> (variant
// 3): 256-wide tiles, so that each A element read by the tensor core and each
// A element split serves twice the columns (a quarter less shared-memory
// traffic per product), on 64-byte rows (64-byte swizzle) to keep 4 raw and 2
// split stages in 192 KiB; 256 tensor-memory columns.
//
// PB (pre-split B): B's TF32 parts come split and transposed from HBM (a
// pass before the kernel), loaded by the TMA straight into the split stages;
// the raw stages hold A only, so 4 raw and 4 split stages fit.
//
// RES (<128, 32> only): A and B of any alignment through residue-class tensor
// maps (res_maps.cuh); the raw stages hold the four class boxes of each
// operand (18 + 16.5 KiB), so 2 raw stages fit beside the 2 split stages.
template <int BN, int BK, bool PB = false, bool RES = false>
struct TcShape {
    static_assert((BN == 128 && BK == 32 && !PB) || (BN == 256 && BK == 16 && !RES), "built shapes");
    static_assert(!RES || (BN == kResTileCols && BK == kResSliceK), "residue-class box geometry");
    static constexpr int kBM = 128;
    static constexpr int kRowBytes = BK * 4;          // one K-major operand row
    static constexpr int kSwizzle = kRowBytes;        // 128- or 64-byte swizzle
    static constexpr int kRawABytes = RES ? 4 * kResAPlaneBytes : kBM * BK * 4;  // TMA A slice, swizzled rows
    static constexpr int kRawBBytes = PB ? 0 : RES ? 4 * kResBPlaneBytes : BK * BN * 4;  // TMA B slice, BN-float rows
    static constexpr int kOpABytes = kBM * BK * 4;    // one K-major A operand tile
    static constexpr int kOpBBytes = BN * BK * 4;     // one K-major B operand tile
    static constexpr int kSplitBytes = 2 * kOpABytes + 2 * kOpBBytes;  // A_big, A_small, B_big, B_small
    static constexpr int kRawStages = RES ? 2 : BK == 32 ? 3 : 4;
    static constexpr int kSplitStages = PB ? 4 : 2;
    static constexpr int kRingBytes = kRawStages * (kRawABytes + kRawBBytes) + kSplitStages * kSplitBytes;
    static constexpr int kSmemBytes = kRingBytes + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr int kTmemCols = BN;
    // Instruction descriptor as kTcIdesc, N = BN.
    static constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                       (static_cast<uint32_t>(kBM >> 4) << 24);
};
static_assert(TcShape<128, 32>::kSmemBytes == kTcSmemBytes, "variant 1 keeps its layout");
static_assert(TcShape<256, 16>::kSmemBytes <= 227 * 1024, "shared memory of variant 3");
static_assert(TcShape<256, 16, true>::kSmemBytes <= 227 * 1024, "shared memory of variant 4");
static_assert(TcShape<128, 32, false, true>::kSmemBytes <= 227 * 1024, "shared memory of variant 1 on class maps");

struct TcParams {
    int M, N, K;
    float* C;
    long long ldc;
    int num_k_tiles;  // ceil(K / BK)
    int tiles_n;      // output tiles per row of tiles
    int tile_base;    // this launch's first tile (split-tile kernels)
    int k_split;      // split-tile kernels, s >= 2: CTAs s t .. s t + s - 1 take
                      // the s parts of the K slices of tile tile_base + t; part 0
                      // stores to C, part q > 0 its partial tile to ws tile
                      // t (s - 1) + q - 1 (128 x BN floats, pitch BN); the CTA
                      // whose arrival on split_count[t] (zero at launch) is the
                      // s-th adds the partial tiles into C in part order
    float* ws;
    unsigned int* split_count;
    int vec_store;    // C base 16-byte aligned and ldc % 4 == 0
    int skip_stage;   // debug: CTA 0's producer never issues K-slice skip_stage-1
    unsigned long long timeout_ns;
    unsigned int* status;
    int a_shift, b_shift;  // residue-class maps: t_j of A's and B's classes (bits 2j, 2j + 1)
};

// ---- "direct-A" variant: the TF32 big part of A is the FP32 tile itself
// (the tensor core reads the top 19 bits of each 32-bit element), so only
// A's small part is stored; B is split into big and small parts and
// transposed to K-major as in the split-tile kernel.  An MMA stage holds the
// raw A slice and the three stored parts and is released by the MMAs; the raw
// B slice has a ring of its own, released as soon as the split warps have
// read it, so that three MMA stages fit.
constexpr int kTdSplitWarps = 8;
constexpr int kTdThreads = 64 + 32 * kTdSplitWarps;
constexpr int kTdBM = 128;
constexpr int kTdBN = 128;
constexpr int kTdBK = 32;
constexpr int kTdTile = 128 * kTdBK * 4;         // 16 KiB: one 128-row x 32-float tile
constexpr int kTdStageBytes = 4 * kTdTile;        // raw A, A small, B big, B small
constexpr int kTdStages = 3;
constexpr int kTdRawBStages = 2;                  // raw B slices
constexpr int kTdRingBytes = kTdStages * kTdStageBytes + kTdRawBStages * kTdTile;
constexpr int kTdSmemBytes = kTdRingBytes + 1024 + 256;
constexpr int kTdTmemCols = kTdBN;

}  // namespace gb300
