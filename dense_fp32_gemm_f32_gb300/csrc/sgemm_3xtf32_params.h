// Tile shape, shared-memory budget, instruction descriptor and kernel
// parameters of the three-product TF32 tensor-core kernel (host and device).
#pragma once

#include <cstdint>

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

struct TcParams {
    int M, N, K;
    float* C;
    long long ldc;
    int num_k_tiles;  // ceil(K / kTcBK)
    int tiles_n;      // output tiles per row of tiles
    int vec_store;    // C base 16-byte aligned and ldc % 4 == 0
    int skip_stage;   // debug: CTA 0's producer never issues K-slice skip_stage-1
    unsigned long long timeout_ns;
    unsigned int* status;
    int dbg;
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
