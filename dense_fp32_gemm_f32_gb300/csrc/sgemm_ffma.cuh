// FP32 matrix multiply on the CUDA cores (FFMA), sm_103a.
//
// C (M x N) = A (M x K) * B (K x N), all row-major float32.
//
// The method is the one the pages build up step by step, re-designed for
// Blackwell:
//  * block tiling with a K sliding window ("Matrix multiplication performance
//    optimisation", section 1 "tiling"): each CTA owns a BM x BN = 128 x 128
//    tile of C and walks K in slices of BK = 32;
//  * shared-memory staging of the A and B slices (same page, section 3) --
//    here written by the Tensor Memory Accelerator (cp.async.bulk.tensor) in
//    one bulk copy per operand instead of by the threads, with the TMA 128-byte
//    swizzle on A in place of the page's "+1" row padding (padding would break
//    the 16-byte alignment of vector loads; the swizzle keeps it and still
//    spreads eight consecutive rows over all banks);
//  * out-of-range elements read as zero (same page, section 3 edge handling):
//    the tensor map's out-of-bounds fill writes zeros, so no load is predicated;
//  * double buffering (same page, section 4) generalised to a STAGES-deep ring
//    of shared-memory slices with a "full" and an "empty" mbarrier per slot.  A
//    dedicated producer warp issues the copies; eight consumer warps compute;
//  * register tiling (same page, section 2; "[infra] 03" experiment 4): every
//    consumer thread accumulates an 8 x 8 block of C in registers and updates
//    it by outer products of 8 A values and 8 B values per k, read from shared
//    memory as 16-byte vectors.  The page reads its 8 A values per k down a
//    column of the A tile; here that per-k read is kept by giving the
//    consumers A with m innermost -- rewritten in shared memory by two
//    transposing warps (kProducerTmaX, the default) or copied transposed in HBM
//    beforehand (AMN) -- so that a thread's 8 rows at one k are two vectors.
//    Reading A as stored (k innermost) instead takes 8 vectors of 4 k values
//    per 4-k group, held for all 4 k, which stalls the first multiply-adds of
//    every group (measured: 82 % FP32-pipe duty against 87-89 %).
//
// Extra machinery not on the pages:
//  * stream-K: one CTA per SM walks whole tiles, then an even share of
//    (tile, K slice) units; tiles shared by several CTAs are finished through
//    a global workspace of partial tiles, in a fixed CTA order;
//  * split-K: for outputs with too few tiles to fill the GPU, a cluster of
//    `split` CTAs along K computes partial tiles over disjoint K ranges and
//    reduces them through distributed shared memory in a fixed rank order
//    (deterministic, no global workspace);
//  * paired FMA (fma.rn.f32x2, sm_100 family): two multiply-adds per
//    instruction, halving the issue slots the outer product needs;
//  * the scaled epilogue of the general entry (SCALED), and the producer
//    variants measured against the default: a cp.async warpgroup (any
//    alignment), a TMA warpgroup with a setmaxnreg register split, a fused
//    producer (4-warp CTAs, two per SM, thread 0 issuing the TMA), 128 x 256
//    tiles.
//
// Every wait is bounded by `timeout_ns` of global time; a thread that gives up
// records SGEMM_ERR_TIMEOUT in the device status word, stops computing, and
// still takes part in every CTA/cluster barrier so that no other thread waits
// forever.  Waits made by whole warps vote, so a warp leaves its loop as one.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "res_maps.cuh"

namespace gb300 {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 32;
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;

enum : int {
    kProducerTma = 1,
    kProducerCpAsync = 2,
    kProducerTmaWg = 3,
    kProducerFused = 4,
    kProducerTmaX = 5,
    kProducerLdg = 7
};

// Producer warps: one elected lane drives the TMA; the cp.async producer
// issues every 4-byte copy itself, so it gets a full warpgroup.
//
// kProducerTmaWg is the TMA producer in a warpgroup of its own, so that the
// CTA is three whole warpgroups (384 threads) and the registers can be split
// between them with setmaxnreg.  At 288 threads (8 consumer warps + 1
// producer warp) one SM sub-partition holds three warps and the allocation
// is capped at 168 registers per thread for every warp; the consumer loop
// wants more (about 230 when unconstrained).  With the split the producer
// warpgroup drops to kRegsProducer and each consumer warp rises to
// kRegsConsumer, which together use exactly the 168 x 384 registers the CTA
// is launched with (setmaxnreg.inc waits until the registers are free, so a
// split that asked for more would never finish: the host launches this
// variant only when the kernel was built with exactly kRegsLaunch).
//
// kProducerFused has no producer warp at all: a CTA of 4 warps that all
// compute (128 x 64 tiles), thread 0 issuing the TMA copies between its own
// multiply-adds, so that two CTAs fit on an SM (2 x 128 threads may use up to
// 255 registers each) and run independently of each other.
//
// kProducerTmaX: the TMA producer warp plus kTransposeWarps transposing
// warps, which copy each stage's A slice (as stored: 128 rows of 32 k) into a
// second slice with m innermost (32 rows of 128 m) for the consumers to read
// per k as two 16-byte vectors (the transposed-A read, without a copy of A in
// HBM).  Two warps, each taking half of the rows, halve the time from a
// slice's arrival to its transposed form (measured on GB300: 4096^3 +1.6 %,
// 1024^3 +4.7 % over one warp); 11 warps leave up to 184 registers a thread.
// kProducerLdg: no tensor maps (operands of any alignment).  Two loader
// warps read A's slice rows from global memory as aligned 16-byte vectors,
// shift each row into place and store it transposed (m innermost), as the
// transposing warps do; two more read B's slice rows the same way and store
// them as they are.  The consumers are those of kProducerTmaX.
// Transposing warps of kProducerTmaX (each rewrites half of the slice's rows).
constexpr int kTransposeWarps = 2;
constexpr int kLoaderWarpsA = 2, kLoaderWarpsB = 2;
// BNK (B stored N x K, k innermost: the general entry's op(B) = B^T read in
// place): one more producer warp transposes each stage's B slice (as loaded:
// 128 rows of 32 k, 128-byte swizzled, the layout of an A slice) into rows of
// k for the consumers.  With the two A-transposing warps that is 12 warps,
// whose 384 threads still get 168 registers each.
constexpr int kTransposeWarpsB = 1;
template <int PRODUCER, bool BNK = false>  // (BNK: any kernel with the B warp, also RES)
__host__ __device__ constexpr int ffma_producer_warps() {
    return (PRODUCER == kProducerFused ? 0
            : PRODUCER == kProducerTma ? 1
            : PRODUCER == kProducerTmaX ? 1 + kTransposeWarps
            : PRODUCER == kProducerLdg  ? kLoaderWarpsA + kLoaderWarpsB
                                        : 4) +
           (BNK ? kTransposeWarpsB : 0);
}
template <int PRODUCER>
__host__ __device__ constexpr int ffma_consumer_warps() {
    return PRODUCER == kProducerFused ? 4 : kConsumerWarps;
}
template <int PRODUCER>
__host__ __device__ constexpr int ffma_min_blocks() {
    return PRODUCER == kProducerFused ? 2 : 1;
}
constexpr int kRegsLaunch = 168;
constexpr int kRegsProducer = 40;
constexpr int kRegsConsumer = 232;
static_assert(4 * 32 * kRegsProducer + kConsumerWarps * 32 * kRegsConsumer == (kConsumerWarps + 4) * 32 * kRegsLaunch,
              "the register split must use exactly the registers the CTA is launched with");
template <int PRODUCER, bool BNK = false>
__host__ __device__ constexpr int ffma_threads() {
    return 32 * (ffma_consumer_warps<PRODUCER>() + ffma_producer_warps<PRODUCER, BNK>());
}
constexpr int kBNWide = 256;  // wide tile: 128 x 256, 8 x 16 per thread (producer warpgroup only)
constexpr int kBNFused = 64;  // 128 x 64 tiles of the fused-producer CTAs
constexpr int kStageABytes = kBM * kBK * 4;      // 16 KiB, 128-byte swizzled rows of 32 floats
// BK = 16 (the tile_k = 16 variant): A slices of 128 rows of 16 floats,
// 64-byte swizzled; B slices of 16 rows.
constexpr int kBK16 = 16;
template <int BK = kBK>
__host__ __device__ constexpr int ffma_stage_a_bytes() {
    return kBM * BK * 4;
}
template <int BN, int BK = kBK>
__host__ __device__ constexpr int ffma_stage_b_bytes() {
    return BK * BN * 4;  // plain rows of BN floats
}
template <int BN, int BK = kBK>
__host__ __device__ constexpr int ffma_stage_bytes() {
    return ffma_stage_a_bytes<BK>() + ffma_stage_b_bytes<BN, BK>();
}
template <int BN>
__host__ __device__ constexpr int ffma_partial_bytes() {
    return kBM * BN * 4;  // one partial tile (split-K, stream-K)
}

// RES (residue-class tensor maps for operands of any alignment): see
// res_maps.cuh; the kernel's tiles are the maps' 128 x 128 tiles with
// 32-deep slices.
static_assert(kResTileRows == kBM && kResTileCols == kBN && kResSliceK == kBK, "residue-class box geometry");
template <bool RES>
struct FfmaMap {
    using type = MapsFor<RES>;
};
// A and B slices as loaded (A slices without RES: kStageABytes; B slices:
// ffma_stage_b_bytes).
template <bool RES, int BK = kBK>
__host__ __device__ constexpr int ffma_load_a_bytes() {
    return RES ? 4 * kResAPlaneBytes : kBM * BK * 4;
}
template <bool RES, int BN, int BK = kBK>
__host__ __device__ constexpr int ffma_load_b_bytes() {
    return RES ? 4 * kResBPlaneBytes : BK * BN * 4;
}

// Thin column edge: when N mod 128 is 1 .. kEdgeMaxCols, those last columns
// are not given a column of tiles of their own (nearly empty tiles that
// would cost as much as full ones); the CTAs working on the last column of
// full tiles compute them too, from the A slices they already hold and the
// edge columns' B values, which an A-transposing warp copies into
// shared memory per slice (kEdgeStageBytes: 32 k x 4 floats).  The
// transposing producer on 32-deep slices, plain epilogue, stream-K only.
constexpr int kEdgeMaxCols = 4;
constexpr int kEdgeStageBytes = kBK * kEdgeMaxCols * 4;
template <int STAGES, bool EDGE>
__host__ __device__ constexpr int ffma_edge_bytes() {
    return EDGE ? STAGES * kEdgeStageBytes : 0;
}

enum : int { kMathFfma = 1, kMathFfma2 = 2 };
enum : unsigned { kStatusTimeout = 4u };

struct FfmaParams {
    int M, N, K;
    const float* A;
    long long lda;
    const float* B;
    long long ldb;
    float* C;
    long long ldc;
    int num_k_tiles;       // ceil(K / BK): K slices
    int split;             // CTAs per cluster along K (== gridDim.z); 1 = no split
    int vec_store;         // C base 16-byte aligned and ldc % 4 == 0
    int tile_base;         // linear index of this launch's first output tile
    int tiles_n;           // output tiles per row of tiles
    int tiles_m;           // rows of output tiles
    int group_m;           // tile order: groups of group_m rows of tiles (1 = row by row; see tile_rc)
    int a_evict_last;      // A's slices are loaded with the L2 evict-last policy
    int b_evict_first;     // B's slices are loaded with the L2 evict-first policy
    int tma_store;         // finished tiles of C go out by tensor-map stores (kernels with a staging tile)
    int c_evict_first;     // those stores carry the L2 evict-first policy
    // Stream-K schedule (sk != 0), one CTA per SM: CTA g first takes whole
    // tiles g, g + G, ... below sk_dp_tiles (data-parallel waves, raster
    // order), then an even share of the units (one K slice of one tile each)
    // of the remaining tiles, dealt out in order; a tile shared by several
    // CTAs is finished by the one holding its first K slice, which adds the
    // others' partial tiles from `ws`.
    int sk;
    int sk_dp_tiles;       // tiles handled whole before the stream-K region
    long long sk_units;    // (tiles - sk_dp_tiles) * num_k_tiles
    float* ws;             // gridDim.x partial tiles of kBM x BN floats
    unsigned int* flags;   // gridDim.x words; flags[g] == sk_seq: CTA g's partial is ready
    unsigned int sk_seq;   // this call's number (nonzero; no flag holds it at launch)
    int skip_stage;        // debug: CTA (0,0,0)'s producer never issues K-slice skip_stage-1
    unsigned long long timeout_ns;
    unsigned int* status;  // per-device sticky status word (error bits)
    // Epilogue of the SCALED kernels: C = alpha * (A B) + beta * C (C is read
    // only when beta != 0).
    float alpha, beta;
    // RES kernels: bits 2j, 2j + 1 hold t_j, the offset in floats of the rows
    // of residue class j inside their 16-byte blocks (res_maps.cuh).
    int a_shift, b_shift;
    // Thin column edge (stream-K launches of the transposing producer with
    // the plain epilogue): ec = N - 128 tiles_n columns, 1 .. kEdgeMaxCols,
    // computed with the last column of tiles (0 = none).  ws_edge: gridDim.x
    // x 256 partial sums (one column pair of one row per consumer thread).
    int ec;
    float2* ws_edge;
};

// Largest dynamic shared memory of a CTA on sm_100-family GPUs.
constexpr int kMaxSmemBytes = 232448;

// XA: the stage also holds the transposed copy of its A slice (kProducerTmaX);
// XB: and of its B slice (BNK).
// RES: the slices as loaded are the residue-class boxes (B is shifted in
// place, so RES needs no XB copy).
template <int STAGES, int BN = kBN, bool XA = false, bool XB = false, int BK = kBK, bool RES = false>
__host__ __device__ constexpr int ffma_ring_bytes() {
    return STAGES * (ffma_load_a_bytes<RES, BK>() + ffma_load_b_bytes<RES, BN, BK>() +
                     (XA ? ffma_stage_a_bytes<BK>() : 0) + (XB ? ffma_stage_b_bytes<BN, BK>() : 0)) >
                   ffma_partial_bytes<BN>()
               ? STAGES * (ffma_load_a_bytes<RES, BK>() + ffma_load_b_bytes<RES, BN, BK>() +
                           (XA ? ffma_stage_a_bytes<BK>() : 0) + (XB ? ffma_stage_b_bytes<BN, BK>() : 0))
               : ffma_partial_bytes<BN>();
}

// The kernels of the transposing producer with the plain epilogue write each
// finished tile of C by a tensor-map store from a staging tile in shared
// memory (when C's base and rows are 16-byte aligned), where it fits.
template <int STAGES, int PRODUCER, int BN, bool SCALED, bool BNK, int BK = kBK, bool RES = false>
__host__ __device__ constexpr bool ffma_tma_store() {
    return (PRODUCER == kProducerTmaX || PRODUCER == kProducerLdg) && BN == kBN && !SCALED &&
           ffma_ring_bytes<STAGES, BN, PRODUCER == kProducerTmaX, BNK, BK, RES>() +
                   ffma_partial_bytes<BN>() + 1024 + 256 +
                   ffma_edge_bytes<STAGES, PRODUCER == kProducerTmaX && !BNK && BK == kBK>() <=
               kMaxSmemBytes;
}

template <int STAGES, int BN = kBN, bool XA = false, bool XB = false, bool STG = false, int BK = kBK,
          bool RES = false, bool EDGE = false>
constexpr int ffma_smem_bytes() {
    return ffma_ring_bytes<STAGES, BN, XA, XB, BK, RES>() + (STG ? ffma_partial_bytes<BN>() : 0) +
           1024 /*align*/ + 256 /*barriers*/ + ffma_edge_bytes<STAGES, EDGE>();
}

// Output tile number -> (row of tiles tm, column of tiles tn).  Tiles are
// numbered in groups of `group_m` rows of tiles, column by column inside a
// group (the last group may hold fewer rows), so that the tiles of one wave
// of CTAs form a block of about group_m x (CTAs / group_m) tiles: each B
// column panel a wave loads then serves group_m tiles instead of one, and
// the group's A row panels serve its consecutive waves.  Odd groups walk
// the columns from the right, so that a group starts on the B panels the
// previous group used last (still in L2).  group_m = 1 is the row-by-row
// order.
__device__ __forceinline__ void tile_rc(int t, int tiles_n, int tiles_m, int group_m, int& tm, int& tn) {
    if (group_m <= 1) {
        tm = t / tiles_n;
        tn = t - tm * tiles_n;
        return;
    }
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int r = t - g * per_group;
    const int rows = min(group_m, tiles_m - g * group_m);
    const int q = r / rows;
    tm = g * group_m + (r - q * rows);
    tn = (g & 1) ? tiles_n - 1 - q : q;
}

// Physical byte offset of float (row r, column c) inside a 128-byte-swizzled
// tile of 32-float rows: the 16-byte chunk index c/4 is XORed with r mod 8.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((((c >> 2) ^ r) & 7) << 4) + (c & 3) * 4);
}

// SCALED: the epilogue applies C = alpha * (A B) + beta * C (FfmaParams
// alpha, beta); a separate instantiation, so that the plain kernels' code is
// not touched by it.
//
// AMN: A is stored transposed (K x M row-major, m innermost: the general
// entry's op(A) = A^T).  The TMA then lands each stage's A slice as 32 rows of
// 128 m values (no swizzle) and a thread reads its 8 rows' values for one k
// as two 16-byte vectors; its rows become wm*32 + 16*(i/4) + 4*tm + i%4.
//
// BNK: B is stored transposed (N x K row-major, k innermost: the general
// entry's op(B) = B^T).  The TMA lands each stage's B slice as 128 rows (n)
// of 32 k with the 128-byte swizzle, and a transposing producer warp rewrites
// it as 32 rows (k) of 128 n, the layout the consumers read.
//
// BK: depth of a K slice, 32 (A slices of 128-byte rows, 128-byte swizzle)
// or 16 (64-byte rows, 64-byte swizzle; the transposing producer on A and B
// as stored only): half the shared memory per stage and twice the slices, so
// that small problems' work divides into finer stream-K units.
//
// RES: A and B of any alignment through residue-class tensor maps
// (res_maps.cuh; tmA and tmB are then four maps each, and FfmaParams
// a_shift, b_shift hold the classes' offsets); the transposing producer,
// 128 x 128 tiles, A and B as stored, 32-deep slices.
//
// EDGE: the thin column edge (FfmaParams ec) is computed with the last
// column of tiles; a separate instantiation, so that the kernels of every
// other shape are compiled without its code.
template <int STAGES, int PRODUCER, int MATH, int BN = kBN, bool SCALED = false, bool AMN = false, bool BNK = false,
          int BK = kBK, bool RES = false, bool EDGE = false>
__global__ void __launch_bounds__(ffma_threads<PRODUCER, BNK || RES>(), ffma_min_blocks<PRODUCER>())
    sgemm_ffma_kernel(const __grid_constant__ typename FfmaMap<RES>::type tmA,
                      const __grid_constant__ typename FfmaMap<RES>::type tmB,
                      const __grid_constant__ CUtensorMap tmC, const FfmaParams p) {
    // 128 accumulators per thread need the consumer register budget of the
    // register split.
    constexpr bool kFused = PRODUCER == kProducerFused;
    static_assert(!AMN || PRODUCER == kProducerTma || PRODUCER == kProducerTmaWg,
                  "transposed A: tensor-map producers only");
    constexpr bool kX = PRODUCER == kProducerTmaX;  // A transposed in shared memory
    static_assert(!(kX && AMN), "A is transposed either in HBM or in shared memory");
    static_assert(!kX || BN == kBN, "in-shared-memory transposition: 128 x 128 tiles");
    constexpr bool kLdg = PRODUCER == kProducerLdg;  // loader warps, no tensor maps
    static_assert(!kLdg || (BN == kBN && !AMN && !BNK && BK == kBK), "loader warps: 128 x 128 tiles, A, B as stored");
    constexpr bool kAT = AMN || kX || kLdg;  // consumers read A with m innermost
    static_assert(!BNK || (BN == kBN && (PRODUCER == kProducerTmaX || (PRODUCER == kProducerTma && AMN))),
                  "B stored N x K: 128 x 128 tiles, transposing producer");
    static_assert(!RES || (kX && BN == kBN && !AMN && !BNK && BK == kBK),
                  "residue-class maps: the transposing producer, 128 x 128 tiles, A, B as stored");
    constexpr int kXA = kX ? kTransposeWarps : 0;          // A-transposing warps
    constexpr int kXB = (BNK || RES) ? kTransposeWarpsB : 0;  // B-transposing (BNK) or B-shifting (RES) warps
    static_assert((BN == kBN && !kFused) || (BN == kBNWide && PRODUCER == kProducerTmaWg) ||
                      (BN == kBNFused && kFused),
                  "tile width");
    static_assert(BK == kBK || (BK == kBK16 && PRODUCER == kProducerTmaX && !BNK && BN == kBN),
                  "16-deep slices: the transposing producer on A and B as stored");
    constexpr int kStageABytes = ffma_stage_a_bytes<BK>();  // (shadows the 32-deep figure)
    constexpr int kStageBBytes = ffma_stage_b_bytes<BN, BK>();
    constexpr int kALoadBytes = ffma_load_a_bytes<RES, BK>();       // A slice as loaded
    constexpr int kBLoadBytes = ffma_load_b_bytes<RES, BN, BK>();   // B slice as loaded
    constexpr int kStageBytes = kALoadBytes + kBLoadBytes;           // bytes the copies of a stage bring
    constexpr int kPartialBytes = ffma_partial_bytes<BN>();
    constexpr int CW = ffma_consumer_warps<PRODUCER>();  // computing warps
    constexpr int CT = 32 * CW;                          // computing threads
    constexpr int WN = kFused ? 1 : 2;                   // warps across the tile's width
    constexpr int H = BN / WN / 32;                      // 4-column groups per thread row (2 or 4)
    constexpr int TQ = 2 * H;                            // column pairs per thread row
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern.
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw_base);
    constexpr int kRingBytes = ffma_ring_bytes<STAGES, BN, kX, BNK, BK, RES>();
    // Staging tile of the tensor-map stores of C, after the ring.
    constexpr bool kStg = ffma_tma_store<STAGES, PRODUCER, BN, SCALED, BNK, BK, RES>();
    constexpr int kStgOff = kRingBytes;
    // Ring: A slices (as loaded), [transposed A slices], B slices (as
    // loaded), [transposed B slices]; with loader warps, transposed A slices
    // and B slices.
    constexpr int kTOff = kLdg ? 0 : STAGES * kALoadBytes;             // transposed A (kX, kLdg)
    constexpr int kBLoadOff = STAGES * kALoadBytes + (kX ? STAGES * kStageABytes : 0);  // B as loaded
    constexpr int kBOff = kBLoadOff + (BNK ? STAGES * kBLoadBytes : 0);  // B as the consumers read it
    constexpr int kBReadStage = BNK ? kStageBBytes : kBLoadBytes;       // its bytes per stage
    // Row k of the B slice the consumers read: rows of BN floats, or (RES)
    // row k / 4 of class k mod 4's box, moved into place.
    auto b_row = [](int k) {
        return RES ? (k & 3) * kResBPlaneBytes + (k >> 2) * (kResBBox * 4) : k * (BN * 4);
    };
    const uint32_t sA0 = base;                                         // STAGES x kALoadBytes
    const uint32_t sB0 = base + kBLoadOff;                             // STAGES x kBLoadBytes
    const uint32_t bar0 = base + kRingBytes + (kStg ? kPartialBytes : 0);  // full[STAGES], empty[STAGES], tfull[STAGES]
    // Thin column edge (FfmaParams ec): B's edge values of each stage, rows of
    // kEdgeMaxCols floats (zeros past N), after the barriers.
    constexpr bool kEdge = EDGE;
    static_assert(!EDGE || (kX && !BNK && BK == kBK && !SCALED), "thin column edge: the transposing producer, "
                                                                  "32-deep slices, plain epilogue");
    constexpr int kEcOff = kRingBytes + (kStg ? kPartialBytes : 0) + 256;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };  // transposed A ready

    constexpr bool kTma = PRODUCER != kProducerCpAsync && !kLdg;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int PW = ffma_producer_warps<PRODUCER>();
    const bool is_producer = !kFused && warp >= CW;
    const int pw = warp - CW;  // producer warp index (when is_producer)
    const int split = p.split;
    const uint32_t crank = split > 1 ? cluster_ctarank() : 0u;

    // Work.  A CTA processes a sequence of segments (tile, kb, ke): the K
    // slices [kb, ke) of one output tile.  Tiles are numbered from tile_base
    // in the grouped order of tile_rc, so that CTAs running at the same time
    // share A row panels and B column panels in L2.  Without stream-K
    // there is one segment: the CTA's tile (gridDim.x over tiles) and, with
    // split-K, the K range of cluster rank blockIdx.z.  With stream-K: the
    // data-parallel tiles first, then the CTA's even share of the stream-K
    // units u (tile = sk_tile0 + u / NK, K slice u % NK).
    const int NK = p.num_k_tiles;
    const int G = static_cast<int>(gridDim.x);
    const int sk_tile0 = p.sk ? p.sk_dp_tiles : p.tile_base + static_cast<int>(blockIdx.x);
    long long u_begin, u_end;
    if (p.sk) {
        u_begin = (p.sk_units * blockIdx.x) / G;
        u_end = (p.sk_units * (blockIdx.x + 1)) / G;
    } else {
        const int kz = (split > 1) ? static_cast<int>(blockIdx.z) : 0;
        u_begin = (static_cast<long long>(NK) * kz) / split;
        u_end = (static_cast<long long>(NK) * (kz + 1)) / split;
    }
    struct Work {
        int dp_next, dp_step, dp_end, tile0, nk;
        long long u, u_end;
        __device__ __forceinline__ bool next(int& tile, int& kb, int& ke) {
            if (dp_next < dp_end) {
                tile = dp_next;
                kb = 0;
                ke = nk;
                dp_next += dp_step;
                return true;
            }
            if (u < u_end) {
                tile = tile0 + static_cast<int>(u / nk);
                kb = static_cast<int>(u % nk);
                ke = static_cast<int>(min(static_cast<long long>(nk), kb + (u_end - u)));
                u += ke - kb;
                return true;
            }
            return false;
        }
    };
    const Work work0{static_cast<int>(blockIdx.x), G, p.sk ? p.sk_dp_tiles : 0, sk_tile0, NK > 0 ? NK : 1,
                     u_begin, NK > 0 ? u_end : u_begin};

    if (threadIdx.x == 0) {
        const uint32_t full_count = kTma ? 1u : 32u * PW;
        // (kX: the transposing warps also release each slot, for its A slice.)
        const uint32_t empty_count = static_cast<uint32_t>(CW + kXA + kXB);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), full_count);
            mbar_init(empty_bar(s), empty_count);
            if (kXA + kXB) mbar_init(tfull_bar(s), 32u * (kXA + kXB));  // every lane of the transposing warps
        }
        fence_mbarrier_init();
    }
    if (kTma && (kFused ? threadIdx.x == 0 : (is_producer && pw == 0 && lane == 0))) {
        if constexpr (RES) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                prefetch_tensormap(&tmA.m[j]);
                prefetch_tensormap(&tmB.m[j]);
            }
        } else {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
        }
    }
    if (split > 1) {
        cluster_sync_all();  // the whole cluster has started before any peer access
    } else {
        __syncthreads();
    }

    bool timed_out = false;
    const unsigned long long tmo = p.timeout_ns;
    const bool skip_here = p.skip_stage > 0 && blockIdx.x == 0 && blockIdx.z == 0;

    // ------------------------------------------------------------ producer
    // The producer and consumer paths never merge again (each ends in its own
    // share of the split-K barriers), so that code after a
    // register-limit change is only reachable through it.
    if (is_producer) {
        // Warpgroup-uniform (warps 8-11).  The producer releases registers
        // first; the consumers' requests are served from what it released.
        if constexpr (PRODUCER == kProducerTmaWg) setmaxnreg_dec<kRegsProducer>();
        const bool issuer = !kLdg && (!kTma || (pw == 0 && lane == 0));
        if constexpr (kLdg) {
            // Loader warps.  pw 0, 1: A's rows 64 pw + lane and 64 pw + 32 +
            // lane of the slice; pw 2, 3: B's rows 16 (pw - 2) .. + 15.  A
            // row's 32 floats of A (B's 128 floats) start at any 4-byte
            // boundary: the lane reads the aligned 16-byte vectors covering
            // them (only those holding an element inside the operand, so
            // nothing outside its rows' extent is touched; the padding and
            // neighbouring elements they also hold are discarded), then
            // picks element j as element sh + j of those vectors, sh = the
            // start's offset in floats within its 16-byte block.  Elements
            // past M, N or K are zeros.  Every lane arrives on the slot's
            // full barrier once its part is stored.
            float* const trA = reinterpret_cast<float*>(smem + kTOff);
            float* const sBp = reinterpret_cast<float*>(smem + kBLoadOff);
            int lit = 0;
            Work lwork = work0;
            int ltile, lkb, lke;
            while (!timed_out && lwork.next(ltile, lkb, lke)) {
                int tm_, tn_;
                tile_rc(ltile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
                const int m0 = tm_ * kBM, n0 = tn_ * BN;
                for (int kt = lkb; kt < lke; ++kt, ++lit) {
                    const int s = lit % STAGES;
                    const int round = lit / STAGES;
                    if (round > 0 && !mbar_wait_bounded_warp(empty_bar(s), (round - 1) & 1, tmo)) {
                        timed_out = true;
                        break;
                    }
                    if (skip_here && lit == p.skip_stage - 1) continue;  // debug: this slice never arrives
                    const int k0 = kt * kBK;
                    const int kval = min(kBK, p.K - k0);  // valid k of the slice (> 0)
                    if (pw < kLoaderWarpsA) {
                        float4 va[2][9];
                        int sh[2];
#pragma unroll
                        for (int qq = 0; qq < 2; ++qq) {
                            const int gm = m0 + lane + 32 * (2 * pw + qq);
                            const bool rin = gm < p.M;
                            const uintptr_t a = reinterpret_cast<uintptr_t>(
                                rin ? p.A + static_cast<long long>(gm) * p.lda + k0 : p.A);
                            const float4* const src = reinterpret_cast<const float4*>(a & ~static_cast<uintptr_t>(15));
                            sh[qq] = static_cast<int>((a >> 2) & 3);
#pragma unroll
                            for (int i = 0; i < 9; ++i) {
                                const int lo = 4 * i - sh[qq];  // offset of the vector's first element
                                va[qq][i] = (rin && lo < kval && lo + 3 >= 0) ? __ldg(src + i)
                                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
                        float* const tr = trA + s * (kStageABytes / 4);
#pragma unroll
                        for (int qq = 0; qq < 2; ++qq) {
                            const int m = lane + 32 * (2 * pw + qq);
                            const int t = sh[qq];
                            auto el = [&](int f) -> float {  // float f of the row's vectors (f static)
                                const float4 v = va[qq][f >> 2];
                                return (f & 3) == 0 ? v.x : (f & 3) == 1 ? v.y : (f & 3) == 2 ? v.z : v.w;
                            };
#pragma unroll
                            for (int j = 0; j < kBK; ++j) {
                                float x = t == 0 ? el(j) : t == 1 ? el(j + 1) : t == 2 ? el(j + 2) : el(j + 3);
                                tr[j * kBM + m] = j < kval ? x : 0.f;
                            }
                        }
                    } else {
                        const int nval = min(BN, p.N - n0);  // valid columns of the tile (> 0)
                        float* const sb = sBp + s * (kStageBBytes / 4);
                        const int c = 4 * lane;
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            float4 v0[8], v1[8];
                            int shb[8];
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                const int kr = 16 * (pw - kLoaderWarpsA) + 8 * half + r;
                                const bool kin = kr < kval;
                                const uintptr_t a = reinterpret_cast<uintptr_t>(
                                    kin ? p.B + static_cast<long long>(k0 + kr) * p.ldb + n0 : p.B);
                                const float4* const src =
                                    reinterpret_cast<const float4*>(a & ~static_cast<uintptr_t>(15));
                                shb[r] = static_cast<int>((a >> 2) & 3);
                                const int lo0 = c - shb[r], lo1 = lo0 + 4;
                                v0[r] = (kin && lo0 < nval && lo0 + 3 >= 0) ? __ldg(src + lane)
                                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                                v1[r] = (kin && shb[r] > 0 && lo1 < nval) ? __ldg(src + lane + 1)
                                                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                const int kr = 16 * (pw - kLoaderWarpsA) + 8 * half + r;
                                const int t = shb[r];
                                const float4 a0 = v0[r], a1 = v1[r];
                                float4 o;
                                o.x = t == 0 ? a0.x : t == 1 ? a0.y : t == 2 ? a0.z : a0.w;
                                o.y = t == 0 ? a0.y : t == 1 ? a0.z : t == 2 ? a0.w : a1.x;
                                o.z = t == 0 ? a0.z : t == 1 ? a0.w : t == 2 ? a1.x : a1.y;
                                o.w = t == 0 ? a0.w : t == 1 ? a1.x : t == 2 ? a1.y : a1.z;
                                if (c + 0 >= nval) o.x = 0.f;
                                if (c + 1 >= nval) o.y = 0.f;
                                if (c + 2 >= nval) o.z = 0.f;
                                if (c + 3 >= nval) o.w = 0.f;
                                *reinterpret_cast<float4*>(sb + kr * BN + c) = o;
                            }
                        }
                    }
                    __syncwarp();
                    mbar_arrive(full_bar(s));  // this lane's part of the slice is stored
                }
            }
        }
        if ((kXA + kXB) > 0 && pw >= 1) {
            // Transposing warps: A slice s (row m: 32 floats in 128-byte
            // swizzled chunks) -> transposed slice (row k: 128 floats); the
            // same for B stored N x K (row n -> row k).  Lane l of an
            // A-transposing warp x takes rows l + 32q for its share of q
            // (x = 0: q = 0, 1; x = 1: q = 2, 3), the B-transposing warp all
            // four q: a 16-byte read of chunk c covers k = 4c..4c+3 of one
            // row (the 8 lanes of each wavefront hit 8 different chunk
            // positions), and each of its 4 floats is stored to row k at
            // column m (or n) (32 consecutive floats per store).
            //
            // RES: the A slice as loaded is four class planes (class j: rows
            // m = 4q + j, q = 0..31, of kResABox floats, the row's element k
            // at t_j + k); see the two branches below.
            const bool xb = (BNK || RES) && pw - 1 >= kXA;  // this warp transposes (RES: shifts) B
            const int qn = xb ? 4 : 4 / kTransposeWarps;
            const int q0 = xb ? 0 : (pw - 1) * qn;
            const int src_off = xb ? kBLoadOff : 0;
            const int dst_off = xb ? kBOff : kTOff;
            // The first A-transposing warp also copies B's thin column edge
            // (FfmaParams ec) for the slices of the last column of tiles: lane
            // l reads row k0 + l's edge values before the slice's wait (their
            // latency overlaps it) and stores them with the transposed slice.
            const bool edge_loader = kEdge && p.ec > 0 && p.sk && pw == 1;
            int xit = 0;
            Work xwork = work0;
            int xtile, xkb, xke;
            while (!timed_out && xwork.next(xtile, xkb, xke)) {
                bool edge_tile = false;
                if (edge_loader) {
                    int tm_, tn_;
                    tile_rc(xtile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
                    edge_tile = tn_ == p.tiles_n - 1;
                }
                for (int kt = xkb; kt < xke; ++kt, ++xit) {
                    const int s = xit % STAGES;
                    const int round = xit / STAGES;
                    float4 eb = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (edge_tile) {
                        const int k = kt * kBK + lane;
                        if (k < p.K) {
                            const float* const brow = p.B + static_cast<long long>(k) * p.ldb + p.tiles_n * kBN;
                            eb.x = __ldg(brow);
                            if (p.ec > 1) eb.y = __ldg(brow + 1);
                            if (p.ec > 2) eb.z = __ldg(brow + 2);
                            if (p.ec > 3) eb.w = __ldg(brow + 3);
                        }
                    }
                    if (!mbar_wait_bounded_warp(full_bar(s), round & 1, tmo)) {
                        timed_out = true;
                        break;
                    }
                    if constexpr (RES) {
                        if (xb) {
                            // In place, a class (8 rows, one t) at a time:
                            // the whole warp reads its rows before any lane
                            // overwrites a vector a neighbour still reads.
                            float* const plane0 = reinterpret_cast<float*>(smem + kBLoadOff + s * kBLoadBytes);
#pragma unroll 1
                            for (int j = 0; j < 4; ++j) {
                                const int t = res_shift(p.b_shift, j);
                                if (t == 0) continue;  // (warp-uniform) already in place
                                float* const plane = plane0 + j * (kResBPlaneBytes / 4) + 4 * lane;
                                float4 o[kBK / 4];
#pragma unroll
                                for (int q = 0; q < kBK / 4; ++q) {
                                    const float4 v0 = *reinterpret_cast<const float4*>(plane + q * kResBBox);
                                    const float4 v1 = *reinterpret_cast<const float4*>(plane + q * kResBBox + 4);
                                    o[q] = t == 1   ? make_float4(v0.y, v0.z, v0.w, v1.x)
                                           : t == 2 ? make_float4(v0.z, v0.w, v1.x, v1.y)
                                                    : make_float4(v0.w, v1.x, v1.y, v1.z);
                                }
                                __syncwarp();
#pragma unroll
                                for (int q = 0; q < kBK / 4; ++q)
                                    *reinterpret_cast<float4*>(plane + q * kResBBox) = o[q];
                            }
                            // These generic-proxy writes precede the slot's
                            // next tensor copy (async proxy) into the same bytes.
                            fence_proxy_async_smem();
                        } else {
                            // Lane l takes rows 4l .. 4l + 3 (row l of each
                            // class plane, 144 bytes apart: the 8 lanes of a
                            // wavefront read 8 different bank groups), warp x
                            // the 4-k groups c = 4x .. 4x + 3: per group and
                            // class two aligned vectors, kept from t_j on (t_j
                            // is the same for the whole warp), then one
                            // 16-byte store of the 4 rows per k.
                            const float* const raw =
                                reinterpret_cast<const float*>(smem + s * kALoadBytes) + lane * kResABox;
                            float* const tr = reinterpret_cast<float*>(smem + kTOff + s * kStageABytes) + 4 * lane;
#pragma unroll
                            for (int cc = 0; cc < kBK / 4 / kTransposeWarps; ++cc) {
                                const int c = (pw - 1) * (kBK / 4 / kTransposeWarps) + cc;
                                float4 r[4];
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const int t = res_shift(p.a_shift, j);
                                    const float* const row = raw + j * (kResAPlaneBytes / 4) + 4 * c;
                                    const float4 v0 = *reinterpret_cast<const float4*>(row);
                                    r[j] = v0;
                                    if (t != 0) {
                                        const float4 v1 = *reinterpret_cast<const float4*>(row + 4);
                                        r[j] = t == 1   ? make_float4(v0.y, v0.z, v0.w, v1.x)
                                               : t == 2 ? make_float4(v0.z, v0.w, v1.x, v1.y)
                                                        : make_float4(v0.w, v1.x, v1.y, v1.z);
                                    }
                                }
                                *reinterpret_cast<float4*>(tr + (4 * c + 0) * kBM) = make_float4(r[0].x, r[1].x, r[2].x, r[3].x);
                                *reinterpret_cast<float4*>(tr + (4 * c + 1) * kBM) = make_float4(r[0].y, r[1].y, r[2].y, r[3].y);
                                *reinterpret_cast<float4*>(tr + (4 * c + 2) * kBM) = make_float4(r[0].z, r[1].z, r[2].z, r[3].z);
                                *reinterpret_cast<float4*>(tr + (4 * c + 3) * kBM) = make_float4(r[0].w, r[1].w, r[2].w, r[3].w);
                            }
                        }
                        if (edge_tile) *reinterpret_cast<float4*>(smem + kEcOff + s * kEdgeStageBytes + 16 * lane) = eb;
                        __syncwarp();
                        mbar_arrive(tfull_bar(s));
                        if (lane == 0) mbar_arrive(empty_bar(s));
                        continue;
                    }
                    const uint8_t* const raw = smem + src_off + s * kStageABytes;
                    float* const tr = reinterpret_cast<float*>(smem + dst_off + s * kStageABytes);
#pragma unroll
                    for (int qq = 0; qq < qn; ++qq) {
                        const int m = lane + 32 * (q0 + qq);
#pragma unroll
                        for (int c = 0; c < BK / 4; ++c) {
                            // 16-byte chunk c of row m: the 128-byte swizzle
                            // XORs the chunk index with m mod 8, the 64-byte
                            // one with (m / 2) mod 4.
                            const int pc = BK == kBK ? ((c ^ m) & 7) : ((c ^ (m >> 1)) & 3);
                            const float4 v = *reinterpret_cast<const float4*>(raw + m * (BK * 4) + (pc << 4));
                            tr[(4 * c + 0) * kBM + m] = v.x;
                            tr[(4 * c + 1) * kBM + m] = v.y;
                            tr[(4 * c + 2) * kBM + m] = v.z;
                            tr[(4 * c + 3) * kBM + m] = v.w;
                        }
                    }
                    if (edge_tile) *reinterpret_cast<float4*>(smem + kEcOff + s * kEdgeStageBytes + 16 * lane) = eb;
                    __syncwarp();
                    mbar_arrive(tfull_bar(s));           // transposed slice written (every lane)
                    if (lane == 0) mbar_arrive(empty_bar(s));  // slice as loaded read
                }
            }
        }
        int issued_round[STAGES];
#pragma unroll
        for (int s = 0; s < STAGES; ++s) issued_round[s] = -1;
        int it = 0;  // K slices so far, across tiles: position in the stage ring
        Work work = work0;
        int tile, kb, ke;
        // With the grouped tile order, the A row panels of a group serve the
        // group's consecutive waves of tiles: loaded evict-last, they stay in
        // L2 while the B column panels stream past.
        const uint64_t a_policy = (kTma && p.a_evict_last) ? l2_policy_evict_last() : 0;
        const uint64_t b_policy = (kTma && p.b_evict_first) ? l2_policy_evict_first() : 0;
        while (issuer && !timed_out && work.next(tile, kb, ke)) {
            int tm_, tn_;
            tile_rc(tile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
            const int n0 = tn_ * BN;
            const int m0 = tm_ * kBM;
            for (int kt = kb; kt < ke; ++kt, ++it) {
                const int s = it % STAGES;
                const int round = it / STAGES;
                const bool ok = kTma ? (round == 0 || mbar_wait_bounded(empty_bar(s), (round - 1) & 1, tmo))
                                     : (round == 0 || mbar_wait_bounded_warp(empty_bar(s), (round - 1) & 1, tmo));
                if (!ok) {
                    timed_out = true;
                    break;
                }
                if (skip_here && it == p.skip_stage - 1) continue;
                const int k0 = kt * BK;
                if (RES) {
                    // Four class boxes per operand (res_maps.cuh): A rows
                    // m0 / 4 .. + 31 of each class from k0; B rows k0 / 4 ..
                    // + 7 of each class from column n0.
                    mbar_arrive_expect_tx(full_bar(s), kStageBytes);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        tma_load_2d(sA0 + s * kALoadBytes + j * kResAPlaneBytes, &res_map(tmA, j), full_bar(s), k0,
                                    m0 >> 2);
                        tma_load_2d(sB0 + s * kBLoadBytes + j * kResBPlaneBytes, &res_map(tmB, j), full_bar(s), n0,
                                    k0 >> 2);
                    }
                } else if (kTma) {
                    mbar_arrive_expect_tx(full_bar(s), kStageBytes);
                    if (AMN) {
                        tma_load_2d(sA0 + s * kStageABytes, &tmA, full_bar(s), m0, k0);
                    } else if (p.a_evict_last) {
                        tma_load_2d_hint(sA0 + s * kStageABytes, &tmA, full_bar(s), k0, m0, a_policy);
                    } else {
                        tma_load_2d(sA0 + s * kStageABytes, &tmA, full_bar(s), k0, m0);
                    }
                    if (BNK) {
                        tma_load_2d(sB0 + s * kStageBBytes, &tmB, full_bar(s), k0, n0);
                    } else if (p.b_evict_first) {
                        tma_load_2d_hint(sB0 + s * kStageBBytes, &tmB, full_bar(s), n0, k0, b_policy);
                    } else {
                        tma_load_2d(sB0 + s * kStageBBytes, &tmB, full_bar(s), n0, k0);
                    }
                } else {
                    // cp.async: PW warps copy 4-byte elements with zero fill;
                    // every lane's copies arrive on the full barrier.
                    const uint32_t sa = sA0 + s * kStageABytes;
                    const uint32_t sb = sB0 + s * kStageBBytes;
                    {  // A slice: 128 rows x 32 floats; lane = column, warp pw
                       // takes rows pw, pw + PW, ...
                        const int k = k0 + lane;
                        const bool kin = k < p.K;
                        for (int r = pw; r < kBM; r += PW) {
                            const int m = m0 + r;
                            const bool in = kin && m < p.M;
                            const float* src = in ? p.A + static_cast<long long>(m) * p.lda + k : p.A;
                            cp_async_4(sa + swz128(r, lane), src, in ? 4u : 0u);
                        }
                    }
                    // B slice: 32 rows x 128 floats; lane = column within a
                    // 32-wide strip, warp pw takes rows pw, pw + PW, ...
                    for (int r = pw; r < BK; r += PW) {
                        const int k = k0 + r;
                        const bool kin = k < p.K;
#pragma unroll
                        for (int q = 0; q < BN / 32; ++q) {
                            const int n = n0 + q * 32 + lane;
                            const bool in = kin && n < p.N;
                            const float* src = in ? p.B + static_cast<long long>(k) * p.ldb + n : p.B;
                            cp_async_4(sb + static_cast<uint32_t>(r * (BN * 4) + (q * 32 + lane) * 4), src,
                                       in ? 4u : 0u);
                        }
                    }
                    cp_async_mbar_arrive_noinc(full_bar(s));
                }
                issued_round[s] = round;
            }
        }
        // Drain: every copy this producer issued has landed before it leaves.
        if (kTma) {
            if (issuer) {
#pragma unroll
                for (int s = 0; s < STAGES; ++s)
                    if (issued_round[s] >= 0 && !mbar_wait_bounded(full_bar(s), issued_round[s] & 1, tmo))
                        timed_out = true;
            }
        } else {
            cp_async_wait_all();
        }
        if (timed_out) atomicOr(p.status, kStatusTimeout);
        // This CTA's share of the barriers at the end of the consumer path.
        if (split > 1) {
            __syncthreads();
            cluster_sync_all();
            cluster_sync_all();
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    if constexpr (PRODUCER == kProducerTmaWg) setmaxnreg_inc<kRegsConsumer>();
    // Warp layout: 4 (M) x 2 (N) warps of 32 x BN/2; each lane owns a 4 x 8
    // grid position (tm, tn).  Thread rows: wm*32 + tm + 4*i (i = 0..7);
    // thread columns: wn*BN/2 + 32*h + tn*4 + {0..3} for h = 0..H-1 (H = 2
    // for the 128-wide tile, 4 for the 256-wide one).  acc[i][q] holds
    // columns (2q, 2q+1) of thread row i, counted over those 4H columns.
    //
    // Per k-group (4 consecutive k) a thread reads 8 A vectors (one per row,
    // 4 k values each: the TMA lands A with k innermost) and, per k, H B
    // vectors, and issues 64 H paired multiply-adds (8 rows x 2H column pairs
    // x 4 k).
    //
    // Lane order.  tm takes lane bits 0 and 2, tn lane bits 1, 3 and 4.
    // Measured on GB300 (shared-memory wavefronts per 16-byte load, ncu): a
    // load whose address changes with both lane bit 0 and lane bit 1 costs 4
    // wavefronts, any other sharing pattern used here costs 2.  With this
    // order neither the A loads (address set by tm) nor the B loads (set by
    // tn) vary with both bits, so every fragment load costs 2 wavefronts
    // instead of 2 (A) and 4 (B) with tn = lane & 7.
    float2 acc[8][TQ];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < TQ; ++q) acc[i][q] = make_float2(0.f, 0.f);  // (K == 0: the empty sum)
    const int wm = kFused ? warp : warp >> 1, wn = kFused ? 0 : warp & 1;
    // Thin column edge (kEdge, FfmaParams ec): in a segment of the last column
    // of tiles, consumer thread (warp, lane) also sums row e_row of the tile
    // times edge columns 2 e_pair and 2 e_pair + 1 (warps 4-7 only when there
    // are more than two), one warp of each SM sub-partition for each pair.
    float2 eacc = make_float2(0.f, 0.f);
    const int e_row = (warp & 3) * 32 + lane;
    const int e_pair = warp >> 2;
    const int tm = (lane & 1) | (((lane >> 2) & 1) << 1);
    const int tn = ((lane >> 1) & 1) | (((lane >> 3) & 1) << 1) | (((lane >> 4) & 1) << 2);

    // Partial tiles (split-K through distributed shared memory, stream-K
    // through global memory) use the layout [e4 = 0..8H-1][thread = 0..255]
    // [4 floats]; element group e4 = i*H + h holds acc[i][2h] and
    // acc[i][2h+1] (four columns).  Consecutive threads touch consecutive 16-byte words, so
    // every partial store and load is conflict-free and coalesced.
    // Output row of the thread's accumulator row i within the tile.
    auto row_in_tile = [&](int i) {
        return kAT ? wm * 32 + 16 * (i >> 2) + 4 * tm + (i & 3) : wm * 32 + tm + 4 * i;
    };

    // C (beta != 0 only): the thread's 8 x H four-column segments of the
    // tile, prefetched into L2 when the CTA starts the segment it will store,
    // so that the epilogue's reads of the old C do not wait on HBM.
    const bool read_c = SCALED && p.beta != 0.f;
    auto prefetch_c = [&](int tile) {
        int tm_, tn_;
        tile_rc(tile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
        const int row0 = tm_ * kBM;
        const int col0 = tn_ * BN + wn * (BN / WN) + tn * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = row0 + row_in_tile(i);
#pragma unroll
            for (int h = 0; h < H; ++h)
                if (r < p.M && col0 + 32 * h < p.N)
                    prefetch_l2(p.C + static_cast<long long>(r) * p.ldc + col0 + 32 * h);
        }
    };
    auto store_c_plain = [&](int tile) {
        int tm_, tn_;
        tile_rc(tile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
        const int row0 = tm_ * kBM;
        const int col0 = tn_ * BN + wn * (BN / WN) + tn * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = row0 + row_in_tile(i);
            if (r >= p.M) continue;
            float* crow = p.C + static_cast<long long>(r) * p.ldc;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const int c = col0 + 32 * h;
                const float4 v =
                    make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y);
                if (p.vec_store && c + 3 < p.N) {
                    *reinterpret_cast<float4*>(crow + c) = v;
                } else {
                    if (c < p.N) crow[c] = v.x;
                    if (c + 1 < p.N) crow[c + 1] = v.y;
                    if (c + 2 < p.N) crow[c + 2] = v.z;
                    if (c + 3 < p.N) crow[c + 3] = v.w;
                }
            }
        }
    };
    auto store_c_scaled = [&](int tile) {
        int tm_, tn_;
        tile_rc(tile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
        const int row0 = tm_ * kBM;
        const int col0 = tn_ * BN + wn * (BN / WN) + tn * 4;
        // Rows in groups of RG: with beta != 0 the group's old C values are
        // all loaded before any of its stores, so the loads are in flight
        // together (a load after a store to C could not be moved above it).
        // The 256-wide tile, short of registers, takes one row at a time.
        constexpr int RG = H == 2 ? 2 : 1;
#pragma unroll
        for (int i0 = 0; i0 < 8; i0 += RG) {
            float4 o[RG][H];
#pragma unroll
            for (int ii = 0; ii < RG; ++ii) {
                const int r = row0 + row_in_tile(i0 + ii);
                const float* crow = p.C + static_cast<long long>(r) * p.ldc;
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const int c = col0 + 32 * h;
                    o[ii][h] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (!read_c || r >= p.M || RG == 1) continue;
                    if (p.vec_store && c + 3 < p.N) {
                        o[ii][h] = *reinterpret_cast<const float4*>(crow + c);
                    } else {
                        if (c < p.N) o[ii][h].x = crow[c];
                        if (c + 1 < p.N) o[ii][h].y = crow[c + 1];
                        if (c + 2 < p.N) o[ii][h].z = crow[c + 2];
                        if (c + 3 < p.N) o[ii][h].w = crow[c + 3];
                    }
                }
            }
#pragma unroll
            for (int ii = 0; ii < RG; ++ii) {
                const int i = i0 + ii;
                const int r = row0 + row_in_tile(i);
                if (r >= p.M) continue;
                float* crow = p.C + static_cast<long long>(r) * p.ldc;
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const int c = col0 + 32 * h;
                    const bool vec = p.vec_store && c + 3 < p.N;
                    float4 v =
                        make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y);
                    {
                        v.x *= p.alpha;
                        v.y *= p.alpha;
                        v.z *= p.alpha;
                        v.w *= p.alpha;
                        if (read_c) {
                            float4 q = o[ii][h];
                            if (RG == 1) {  // loaded here, just before its store
                                if (vec) {
                                    q = *reinterpret_cast<const float4*>(crow + c);
                                } else {
                                    if (c < p.N) q.x = crow[c];
                                    if (c + 1 < p.N) q.y = crow[c + 1];
                                    if (c + 2 < p.N) q.z = crow[c + 2];
                                    if (c + 3 < p.N) q.w = crow[c + 3];
                                }
                            }
                            v.x = fmaf(p.beta, q.x, v.x);
                            v.y = fmaf(p.beta, q.y, v.y);
                            v.z = fmaf(p.beta, q.z, v.z);
                            v.w = fmaf(p.beta, q.w, v.w);
                        }
                    }
                    if (vec) {
                        *reinterpret_cast<float4*>(crow + c) = v;
                    } else {
                        if (c < p.N) crow[c] = v.x;
                        if (c + 1 < p.N) crow[c + 1] = v.y;
                        if (c + 2 < p.N) crow[c + 2] = v.z;
                        if (c + 3 < p.N) crow[c + 3] = v.w;
                    }
                }
            }
        }
    };
    auto consumer_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(CT) : "memory"); };
    // Tensor-map store of a finished tile: the consumers write it into the
    // staging tile (row-major, BN floats a row: a warp's 16-byte stores take
    // the minimum 4 wavefronts, its lanes' four rows landing on the same
    // banks 8 lanes at a time), then one thread hands it to the TMA and the
    // consumers go on to their next tile while it is written out; the TMA
    // clips the rows and columns outside C.  Before the staging tile is
    // written again, that thread waits until the previous store has read it.
    auto store_c_tma = [&](int tile) {
        int tm_, tn_;
        tile_rc(tile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
        float* const stg = reinterpret_cast<float*>(smem + kStgOff);
        if (threadIdx.x == 0) bulk_wait_read_all();
        consumer_sync();
        const int col0 = wn * (BN / WN) + tn * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int h = 0; h < H; ++h)
                *reinterpret_cast<float4*>(stg + row_in_tile(i) * BN + col0 + 32 * h) =
                    make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y);
        fence_proxy_async_smem();  // the generic-proxy writes, visible to the TMA
        consumer_sync();
        if (threadIdx.x == 0) {
            if (p.c_evict_first)
                tma_store_2d_hint(&tmC, smem_addr(stg), tn_ * BN, tm_ * kBM, l2_policy_evict_first());
            else
                tma_store_2d(&tmC, smem_addr(stg), tn_ * BN, tm_ * kBM);
            bulk_commit_group();
        }
    };
    // C whose rows are not 16-byte addressable (a base or ldc off the
    // 16-byte grid): the consumers stage the finished tile as for the
    // tensor-map store, then write it out row by row, consumer warp w taking
    // rows w, w + 8, ... and lane l the columns l, l + 32, l + 64, l + 96 of
    // each, so that every store instruction writes 128 consecutive bytes
    // (the 4-byte stores of the threads' own blocks write 4 rows x 8 groups
    // of 4 floats an instruction).  Measured on GB300: 1023 x 1025 x 1027
    // 56.4 us with C's rows of 1025 floats, 53.7 with the same rows padded to
    // 1028 (16-byte stores).
    auto store_c_rows = [&](int tile) {
        int tm_, tn_;
        tile_rc(tile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
        float* const stg = reinterpret_cast<float*>(smem + kStgOff);
        consumer_sync();  // every row of the previous tile has been read
        const int col0 = wn * (BN / WN) + tn * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int h = 0; h < H; ++h)
                *reinterpret_cast<float4*>(stg + row_in_tile(i) * BN + col0 + 32 * h) =
                    make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y);
        consumer_sync();
        const int row0 = tm_ * kBM, c0 = tn_ * BN;
        const int nval = min(BN, p.N - c0);
        for (int r = warp; r < kBM && row0 + r < p.M; r += CW) {
            float* const crow = p.C + static_cast<long long>(row0 + r) * p.ldc + c0;
            const float* const srow = stg + r * BN;
#pragma unroll
            for (int c = lane; c < BN; c += 32)
                if (c < nval) crow[c] = srow[c];
        }
    };
    auto store_c = [&](int tile) {
        if constexpr (SCALED) {
            store_c_scaled(tile);
        } else if constexpr (kStg) {
            if (p.tma_store) {
                store_c_tma(tile);
            } else if (!p.vec_store) {
                store_c_rows(tile);
            } else {
                store_c_plain(tile);
            }
        } else {
            store_c_plain(tile);
        }
    };
    // The thread's finished edge sums (kEdge): row e_row of the tile, columns
    // 128 tiles_n + 2 e_pair (+ 1 when that is inside C).
    auto store_edge = [&](int tile) {
        int tm_, tn_;
        tile_rc(tile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
        const int r = tm_ * kBM + e_row;
        if (r >= p.M) return;
        float* const ce = p.C + static_cast<long long>(r) * p.ldc + p.tiles_n * kBN + 2 * e_pair;
        ce[0] = eacc.x;
        if (2 * e_pair + 1 < p.ec) ce[1] = eacc.y;
    };
    // The TMA has finished the last store of this CTA (reading the staging
    // tile and writing C) before the CTA's shared memory is released.
    auto drain_stores = [&] {
        if constexpr (kStg)
            if (p.tma_store && threadIdx.x == 0) bulk_wait_all();
    };

    {
        // Byte offsets inside a stage.  A row r = wm*32 + tm + 4i has r mod 8 =
        // tm + 4*(i & 1), so even i share one swizzle key and odd i the other.
        const uint32_t a_row0 = kAT ? static_cast<uint32_t>((kX ? kTOff : 0) + (wm * 32 + 4 * tm) * 4)
                                    : static_cast<uint32_t>((wm * 32 + tm) * 128);
        const uint32_t b_col0 = static_cast<uint32_t>((wn * (BN / WN) + tn * 4) * 4);
        const uint8_t* const smem_a = smem + a_row0;                          // generic pointers
        const uint8_t* const smem_b = smem + kBOff + b_col0;  // for the vector loads

        // Fused producer (thread 0 of a kProducerFused CTA): the loads follow
        // the same work sequence as the computation.  STAGES loads go out
        // before the first K slice; at the start of K slice it (> 0) the slot
        // of slice it-1 is refilled with load it-1+STAGES, once every warp has
        // released it (usually already: the warps run side by side).
        Work lwork = work0;
        int ltile = 0, lkb = 0, lke = 0, lkt = 0, loads = 0;
        bool lhave = false, lfail = false;
        auto issue_load = [&]() {
            if (!lhave || lfail) return;
            const int s = loads % STAGES;
            const int round = loads / STAGES;
            if (round > 0 && !mbar_wait_bounded(empty_bar(s), (round - 1) & 1, tmo)) {
                lfail = true;  // the consumers' own bounded waits then end the loop
                return;
            }
            if (!(skip_here && loads == p.skip_stage - 1)) {
                const int k0 = lkt * BK;
                mbar_arrive_expect_tx(full_bar(s), kStageBytes);
                int tm_, tn_;
                tile_rc(ltile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
                tma_load_2d(sA0 + s * kStageABytes, &tmA, full_bar(s), k0, tm_ * kBM);
                tma_load_2d(sB0 + s * kStageBBytes, &tmB, full_bar(s), tn_ * BN, k0);
            }
            ++loads;
            if (++lkt >= lke) {
                lhave = lwork.next(ltile, lkb, lke);
                lkt = lkb;
            }
        };
        if (kFused && threadIdx.x == 0) {
            lhave = lwork.next(ltile, lkb, lke);
            lkt = lkb;
            for (int j = 0; j < STAGES; ++j) issue_load();
        }

        int it = 0;
        Work work = work0;
        int tile, kb, ke;
        while (!timed_out && work.next(tile, kb, ke)) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < TQ; ++q) acc[i][q] = make_float2(0.f, 0.f);
            bool e_work = false;  // (warp-uniform)
            if (kEdge && p.ec > 0 && p.sk) {
                int tm_, tn_;
                tile_rc(tile, p.tiles_n, p.tiles_m, p.group_m, tm_, tn_);
                e_work = tn_ == p.tiles_n - 1 && 2 * e_pair < p.ec;
            }
            eacc = make_float2(0.f, 0.f);
            if (SCALED && read_c && kb == 0 && (split <= 1 || crank == 0))
                prefetch_c(tile);  // this CTA stores the tile

            for (int kt = kb; kt < ke; ++kt, ++it) {
                const int s = it % STAGES;
                const int round = it / STAGES;
                if (kFused && threadIdx.x == 0 && it > 0) issue_load();
                if (!mbar_wait_bounded_warp(full_bar(s), round & 1, tmo) ||
                    ((kXA + kXB) > 0 && !mbar_wait_bounded_warp(tfull_bar(s), round & 1, tmo))) {
                    timed_out = true;
                    break;
                }
                const uint8_t* sa = smem_a + s * kStageABytes;
                const uint8_t* sb = smem_b + s * kBReadStage;
#pragma unroll
                for (int kg = 0; kg < BK / 4; ++kg) {
                    const uint32_t xe = static_cast<uint32_t>(((kg ^ tm) & 7) << 4);
                    const uint32_t xo = xe ^ 64u;
                    float4 a[8];
                    if (!kAT) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            a[i] = *reinterpret_cast<const float4*>(sa + i * 512 + ((i & 1) ? xo : xe));
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int k = kg * 4 + kk;
                        float am[8];  // kAT: rows 4*tm + {0..3} and 16 + 4*tm + {0..3} at this k
                        if (kAT) {
                            const float4 a0 = *reinterpret_cast<const float4*>(sa + k * (kBM * 4));
                            const float4 a1 = *reinterpret_cast<const float4*>(sa + k * (kBM * 4) + 64);
                            am[0] = a0.x, am[1] = a0.y, am[2] = a0.z, am[3] = a0.w;
                            am[4] = a1.x, am[5] = a1.y, am[6] = a1.z, am[7] = a1.w;
                        }
                        float2 bp[TQ];
#pragma unroll
                        for (int h = 0; h < H; ++h) {
                            const float4 bv = *reinterpret_cast<const float4*>(sb + b_row(k) + h * 128);
                            bp[2 * h] = make_float2(bv.x, bv.y);
                            bp[2 * h + 1] = make_float2(bv.z, bv.w);
                        }
                        // Column pair outermost: each B pair feeds 8 consecutive
                        // multiply-adds (measured faster than row-outermost order).
#pragma unroll
                        for (int q = 0; q < TQ; ++q)
#pragma unroll
                            for (int i0 = 0; i0 < 8; ++i0) {
                                const int i = (q & 1) ? 7 - i0 : i0;  // serpentine: A value reused across q
                                const float av = kAT        ? am[i]
                                                 : kk == 0 ? a[i].x
                                                 : kk == 1 ? a[i].y
                                                 : kk == 2 ? a[i].z
                                                           : a[i].w;
                                if (MATH == kMathFfma2) {
                                    acc[i][q] = __ffma2_rn(make_float2(av, av), bp[q], acc[i][q]);
                                } else {
                                    acc[i][q].x = fmaf(av, bp[q].x, acc[i][q].x);
                                    acc[i][q].y = fmaf(av, bp[q].y, acc[i][q].y);
                                }
                            }
                    }
                }
                if (kEdge && e_work) {
                    // The edge columns' sums over this slice: A's row e_row at
                    // each k (the transposed slice: 32 lanes, 128 consecutive
                    // bytes) times the pair's B values (one broadcast); two
                    // chains of 16 k.
                    const float* const ta = reinterpret_cast<const float*>(smem + kTOff + s * kStageABytes) + e_row;
                    const float2* const eb =
                        reinterpret_cast<const float2*>(smem + kEcOff + s * kEdgeStageBytes) + e_pair;
                    float2 e0 = make_float2(0.f, 0.f), e1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < kBK; k += 2) {
                        const float a0 = ta[k * kBM], a1 = ta[(k + 1) * kBM];
                        const float2 b0 = eb[2 * k], b1 = eb[2 * (k + 1)];
                        e0 = __ffma2_rn(make_float2(a0, a0), b0, e0);
                        e1 = __ffma2_rn(make_float2(a1, a1), b1, e1);
                    }
                    eacc.x += e0.x + e1.x;
                    eacc.y += e0.y + e1.y;
                }
                // Every load from stage s has returned (its values were
                // consumed above): release the slot to the producer(s).
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
            }
            if (!p.sk || timed_out) break;  // one tile per CTA; its epilogue follows below

            // ---------------------------------------------------- stream-K epilogue
            float* const ws_mine = p.ws + static_cast<size_t>(blockIdx.x) * (kBM * BN);
            if (kb > 0) {
                // Not the first K slice of the tile: leave the partial tile for
                // the CTA that holds the first slice.
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        __stcg(reinterpret_cast<float4*>(ws_mine) + (i * H + h) * CT + threadIdx.x,
                               make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                                           acc[i][2 * h + 1].y));
                if (e_work) __stcg(p.ws_edge + static_cast<size_t>(blockIdx.x) * CT + threadIdx.x, eacc);
                consumer_sync();
                if (threadIdx.x == 0) {
                    __threadfence();
                    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.flags + blockIdx.x), "r"(p.sk_seq)
                                 : "memory");
                }
            } else {
                if (ke < NK) {
                    // First slice but not the whole K range: add the partial
                    // tiles of the CTAs whose runs start inside this tile, in
                    // CTA order (a fixed order: deterministic sums).
                    const long long tile_end = static_cast<long long>(tile - sk_tile0 + 1) * NK;  // in units
                    for (long long g2 = blockIdx.x + 1; g2 < G && (p.sk_units * g2) / G < tile_end; ++g2) {
                        bool ok = true;
                        if (threadIdx.x == 0) {
                            const uint64_t t0 = global_timer_ns();
                            unsigned int f = 0;
                            while (true) {
                                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
                                             : "=r"(f)
                                             : "l"(p.flags + g2)
                                             : "memory");
                                if (f == p.sk_seq) break;
                                if (global_timer_ns() - t0 > tmo) {
                                    ok = false;
                                    break;
                                }
                            }
                            if (!ok) atomicOr(p.status, kStatusTimeout);
                        }
                        consumer_sync();  // thread 0 saw the flag: the partial is complete
                        const float4* src = reinterpret_cast<const float4*>(p.ws + g2 * (kBM * BN));
#pragma unroll
                        for (int i = 0; i < 8; ++i)
#pragma unroll
                            for (int h = 0; h < H; ++h) {
                                const float4 v = __ldcg(src + (i * H + h) * CT + threadIdx.x);
                                acc[i][2 * h].x += v.x;
                                acc[i][2 * h].y += v.y;
                                acc[i][2 * h + 1].x += v.z;
                                acc[i][2 * h + 1].y += v.w;
                            }
                        if (e_work) {
                            const float2 v = __ldcg(p.ws_edge + static_cast<size_t>(g2) * CT + threadIdx.x);
                            eacc.x += v.x;
                            eacc.y += v.y;
                        }
                    }
                }
                store_c(tile);
                if (e_work) store_edge(tile);
            }
        }
        if (kFused && threadIdx.x == 0) {
            // Loads still in flight (the loop ended early): let them land
            // before the CTA's shared memory is released.  Slot j % STAGES
            // holds no later load than j, so phase parity (j / STAGES) & 1
            // identifies its completion.
            for (int j = loads > STAGES ? loads - STAGES : 0; j < loads; ++j)
                if (j >= it && !(skip_here && j == p.skip_stage - 1) &&
                    !mbar_wait_bounded(full_bar(j % STAGES), (j / STAGES) & 1, tmo))
                    timed_out = true;
            if (lfail) timed_out = true;
        }
        if (timed_out) atomicOr(p.status, kStatusTimeout);
    }

    // ------------------------------------------------------------ split-K reduction
    if (split > 1) {
        // All consumer reads of the ring are finished once every thread of the
        // CTA passes this barrier; the ring is then reused for the partial tile.
        __syncthreads();
        if (crank != 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int h = 0; h < H; ++h)
                    sts128(base + static_cast<uint32_t>(((i * H + h) * CT + threadIdx.x) * 16),
                           make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y));
        }
        cluster_sync_all();
        if (crank == 0) {
            for (int r = 1; r < split; ++r) {  // fixed order: deterministic sums
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const uint32_t off =
                            base + static_cast<uint32_t>(((i * H + h) * CT + threadIdx.x) * 16);
                        const float4 v = ld_shared_cluster_v4(map_shared_rank(off, static_cast<uint32_t>(r)));
                        acc[i][2 * h].x += v.x;
                        acc[i][2 * h].y += v.y;
                        acc[i][2 * h + 1].x += v.z;
                        acc[i][2 * h + 1].y += v.w;
                    }
            }
        }
        cluster_sync_all();  // peers keep their shared memory alive until rank 0 has read it
        if (crank != 0) return;
    }

    if (p.sk) {  // (stream-K CTAs stored their tiles above)
        drain_stores();
        return;
    }

    // ------------------------------------------------------------ epilogue
    store_c(p.tile_base + static_cast<int>(blockIdx.x));
    drain_stores();
}

}  // namespace gb300
