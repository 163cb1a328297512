// The three-product TF32 entries' work: variant choice, the pass splitting B,
// and the launches (sgemm_3xtf32, sgemm_3xtf32_ex).
#include "api_internal.h"

namespace gb300 {
namespace detail {

int run_3xtf32(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
               void* stream, const sgemm_options* opt) {
    int rc = validate(M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (opt && opt->debug_skip_stage < 0) return SGEMM_ERR_INVALID_ARG;
    // Forced K split: 1 = none, 2..4 = CTAs per tile (variant 1); for
    // variants 3 and 4, 2 = split the last partial wave's tiles whatever K.
    const int force_s = opt ? opt->split_k : 0;
    if (force_s < 0 || force_s > 4) return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    int dev = 0;
    DeviceState* st = nullptr;
    rc = current_device(&dev, &st);
    if (rc != SGEMM_OK) return rc;
    // The tensor-core kernels are fed by tensor maps.  Operands the TMA
    // cannot read directly (unaligned bases or row strides) go to the
    // split-tile kernel on residue-class maps (variant 1's tiles; M, K >= 4)
    // when that is the variant anyway or the product is below 2^30 flop;
    // larger products for the wide-tile variants are repacked into pitched
    // rows first.  K == 0, and misaligned operands neither path takes, run
    // the FFMA kernel, which meets the same contract.
    // Variant: 1 = split-tile kernel (all four TF32 parts in shared memory),
    // 2 = direct-A kernel (A's big part is the TMA tile itself), 3 = the
    // split-tile kernel on 128 x 256 tiles with K-slices of 16, 4 = variant
    // 3 with B's TF32 parts split and transposed in HBM by a pass before the
    // kernel (one read of B and two writes of its size), which leaves the
    // kernel's split warps A only.  Automatic: 4 when the 128 x 256 tiles
    // number at least half the SMs and M >= 1024 (the pass costs ~6/M bytes
    // per flop), 3 when they do with fewer rows, else 1.  Measured on GB300,
    // TFLOP/s for 1 / 3 / 4: 2048^3 152 / 181 / 205, 4096^3 195 / 221 / 274,
    // 8192^3 208 / 246 / 289, 4096 x 4096 x 256 99 / 112 / 117; with fewer
    // tiles (variant 1 with its K split, below) 1024^3 72 / 40 / 46, 8192 x
    // 128 x 8192 148 / 51 / 70, 128 x 8192 x 16384 162 / 54 / 23.
    int variant = (opt && opt->math) ? opt->math : 0;
    if (variant == 0)
        variant = 2 * ceil_div(M, kTcBM) * ceil_div(N, 256) < st->sm_count ? 1 : M >= 1024 ? 4 : 3;
    if (variant < 1 || variant > 4 || (force_s >= 2 && variant == 2) || (force_s >= 3 && variant >= 3))
        return SGEMM_ERR_INVALID_ARG;
    if (force_s >= 2 && force_s > ceil_div(K, kTcBK)) return SGEMM_ERR_INVALID_ARG;  // a slice per part at least
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int misaligned = (tma_ok(A, lda) ? 0 : 1) | (tma_ok(B, ldb) ? 0 : 2);
    const double flops = 2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K);
    const bool variant_forced = opt && opt->math;
    bool res = false;  // the residue-class maps (variant 1's kernel on them)
    if (K >= 4 && M >= 4 && misaligned && (variant == 1 || (!variant_forced && flops < kRepackMinFlops))) {
        res = true;
        variant = 1;
    }
    Repacked packed;
    if (!res && K > 0 && misaligned && flops >= kRepackMinFlops)
        (void)packed.make(dev, *st, misaligned, M, N, K, A, lda, B, ldb, cs);  // (on failure: the FFMA kernel)
    if (K == 0 || (!res && (!tma_ok(A, lda) || !tma_ok(B, ldb)))) {
        packed.release();
        return run_ffma(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr);
    }
    // Launches: (kernel, tile width, K-slice, grid, first tile, K split).
    // Variants 3 and 4 run whole waves of 128 x 256 tiles; the tiles of a
    // last partial wave run in a second launch of the same kernel with their K
    // slices split between two CTAs each (twice the CTAs at half the work: a
    // fuller wave), the second halves' partial tiles added into C by the
    // tile's CTA that finishes last (in part order: deterministic).  4096^3:
    // 3 waves of 152 wide tiles, then 112 CTAs on the last 56 (262 -> 277
    // TFLOP/s).  Only for K >= kTcTailSplitMinK: with shorter K the halves'
    // pipeline fill and the partial tiles' traffic cost more than the fuller
    // wave gains (figures beside the constant), and the tiles run as one
    // launch.
    struct TcLaunch {
        KernelEntry k;
        int bn, bk;
        long long grid;
        int tile_base, k_split;
        bool pb;  // B's TF32 parts pre-split in HBM (variant 4)
    };
    TcLaunch launches[2];
    int nl = 1;
    const long long tiles_m = ceil_div(M, kTcBM);
    // The launch whose tiles are split along K (if any): split_s parts per
    // tile, split_tiles tiles of width split_bn.
    int split_l = -1, split_s = 1, split_bn = 0;
    long long split_tiles = 0;
    if (variant >= 3) {
        const KernelEntry wk = variant == 4 ? tf32x3_wide_pb_kernel() : tf32x3_wide_kernel();
        const bool pb = variant == 4;
        const long long wide = tiles_m * ceil_div(N, 256);
        const long long full = (wide / st->sm_count) * st->sm_count;
        const bool want_split = force_s == 2 || (force_s == 0 && K >= kTcTailSplitMinK);
        if (full > 0 && full < wide && want_split && ceil_div(K, 16) >= 2) {
            split_l = 1, split_s = 2, split_bn = 256, split_tiles = wide - full;
            launches[0] = {wk, 256, 16, full, 0, 0, pb};
            launches[1] = {wk, 256, 16, split_s * split_tiles, static_cast<int>(full), split_s, pb};
            nl = 2;
        } else {
            launches[0] = {wk, 256, 16, wide, 0, 0, pb};
        }
    } else {
        const KernelEntry k = res ? tf32x3_res_kernel() : variant == 1 ? tf32x3_kernel() : tf32x3_direct_kernel();
        const long long tiles = tiles_m * ceil_div(N, kTcBN);
        // Variant 1 with at most half as many tiles as SMs: each tile's nk K
        // slices split among s = min(4, SMs / tiles, nk / 2) CTAs when the
        // slices that takes off each CTA, nk (s - 1) / s, outnumber the
        // split's cost, measured as about 7 + 2 (s - 1) slices of one CTA (the
        // counters' reset, each part's pipeline fill, the partial tiles
        // written, read and added).  Measured, TFLOP/s without / with: 1024^3
        // (s = 2) 61 / 71, 1024^2 x 768 55 / 61, 1024^2 x 2048 72 / 101, 768^3
        // (s = 4) 31 / 34, 8192 x 128 x 8192 85 / 148, 128 x 8192 x 16384 89 /
        // 165; 1024^2 x 512 46 / 44, 512^3 12.1 / 11.6 and 256^3 2.0 / 1.6
        // stay whole.
        const long long nk = ceil_div(K, kTcBK);
        long long s = 1;
        if (force_s >= 1) {
            s = force_s;
        } else if (variant == 1 && 2 * tiles <= st->sm_count) {
            s = std::min<long long>({4, st->sm_count / tiles, nk / 2});
            if (s >= 2 && nk * (s - 1) < s * (7 + 2 * (s - 1))) s = 1;
        }
        if (s >= 2) {
            split_l = 0, split_s = static_cast<int>(s), split_bn = kTcBN, split_tiles = tiles;
            launches[0] = {k, kTcBN, kTcBK, split_s * tiles, 0, split_s, false};
        } else {
            launches[0] = {k, kTcBN, kTcBK, tiles, 0, 0, false};
        }
    }
    // The later parts' partial tiles (128 x split_bn floats each) and a
    // counter of arrived parts per split tile (zeroed here), from the pool.
    void* ws_split = nullptr;
    unsigned int* split_count = nullptr;
    if (split_l >= 0) {
        cudaMemPool_t pool = workspace_pool(dev, *st);
        const size_t part_bytes =
            (static_cast<size_t>(split_tiles) * (split_s - 1) * kTcBM * split_bn * sizeof(float) + 255) &
            ~size_t{255};
        const size_t count_bytes = static_cast<size_t>(split_tiles) * sizeof(unsigned int);
        if (!pool || cudaMallocFromPoolAsync(&ws_split, part_bytes + count_bytes, pool, cs) != cudaSuccess) {
            (void)cudaGetLastError();
            packed.release();
            return SGEMM_ERR_CUDA;
        }
        split_count = reinterpret_cast<unsigned int*>(static_cast<char*>(ws_split) + part_bytes);
        if (cudaMemsetAsync(split_count, 0, count_bytes, cs) != cudaSuccess) {
            (void)cudaGetLastError();
            (void)cudaFreeAsync(ws_split, cs);
            packed.release();
            return SGEMM_ERR_CUDA;
        }
    }

    // Variant 4: B's TF32 parts, transposed (N x Kp), in a pool buffer.  Rows
    // of Kp = K rounded up to 32 floats start on 128-byte boundaries, so that
    // each 64-byte box row the TMA reads lies in one 128-byte line (measured
    // on GB300, 4096 x 4096 x 4099: 818 us with rows of K rounded up to 4
    // floats, against 499 us at K = 4096).
    void* ws = nullptr;
    float *bt_big = nullptr, *bt_small = nullptr;
    const long long Kp = (static_cast<long long>(K) + 31) / 32 * 32;
    const size_t part = (static_cast<size_t>(N) * Kp * sizeof(float) + 255) & ~size_t{255};
    if (launches[0].pb) {
        cudaMemPool_t pool = workspace_pool(dev, *st);
        if (!pool || cudaMallocFromPoolAsync(&ws, 2 * part, pool, cs) != cudaSuccess) {
            // No room for B's parts (2 N K floats): variant 3's kernels, which
            // split B in shared memory, on the same tiles.
            (void)cudaGetLastError();
            ws = nullptr;
            for (int l = 0; l < nl; ++l) {
                launches[l].k = tf32x3_wide_kernel();
                launches[l].pb = false;
            }
        }
    }
    if (launches[0].pb) {
        bt_big = static_cast<float*>(ws);
        bt_small = reinterpret_cast<float*>(static_cast<char*>(ws) + part);
        rc = split_transpose_b(B, ldb, K, N, bt_big, bt_small, Kp, cs);
        if (rc != SGEMM_OK) {
            (void)cudaFreeAsync(ws, cs);
            if (ws_split) (void)cudaFreeAsync(ws_split, cs);
            packed.release();
            return rc;
        }
    }

    rc = SGEMM_OK;
    for (int l = 0; l < nl && rc == SGEMM_OK; ++l) {
        const TcLaunch& ln = launches[l];
        alignas(64) CUtensorMap tmA;
        alignas(64) CUtensorMap tmB;
        alignas(64) CUtensorMap tmB2;
        std::memset(&tmB2, 0, sizeof tmB2);
        ResMaps resA, resB;  // (res) boxes of 36 k x 32 rows of A, 132 columns x 8 rows of B
        int a_shift = 0, b_shift = 0;
        const CUtensorMapSwizzle swz = ln.bk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        if (res) {
            rc = encode_res(&resA, &a_shift, A, M, K, lda, kResABox, kResTileRows / 4);
            if (rc == SGEMM_OK) rc = encode_res(&resB, &b_shift, B, K, N, ldb, kResBBox, kResSliceK / 4);
        } else {
            rc = encode_2d(&tmA, A, K, M, lda, ln.bk, kTcBM, swz);
            if (ln.pb) {  // {k, n} boxes of the transposed parts, swizzled like A
                if (rc == SGEMM_OK) rc = encode_2d(&tmB, bt_big, K, N, Kp, ln.bk, ln.bn, swz);
                if (rc == SGEMM_OK) rc = encode_2d(&tmB2, bt_small, K, N, Kp, ln.bk, ln.bn, swz);
            } else {
                if (rc == SGEMM_OK) rc = encode_2d(&tmB, B, N, K, ldb, ln.bn, ln.bk, CU_TENSOR_MAP_SWIZZLE_NONE);
                tmB2 = tmB;  // (unused)
            }
        }
        if (rc != SGEMM_OK) break;

        TcParams prm;
        prm.M = M;
        prm.N = N;
        prm.K = K;
        prm.C = C;
        prm.ldc = ldc;
        prm.num_k_tiles = static_cast<int>(ceil_div(K, ln.bk));
        prm.tiles_n = static_cast<int>(ceil_div(N, ln.bn));
        prm.tile_base = ln.tile_base;
        prm.k_split = ln.k_split;
        prm.ws = ln.k_split > 1 ? static_cast<float*>(ws_split) : nullptr;
        prm.split_count = ln.k_split > 1 ? split_count : nullptr;
        prm.vec_store = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0) ? 1 : 0;
        prm.skip_stage = opt ? opt->debug_skip_stage : 0;
        prm.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
        prm.status = st->status_word;
        prm.a_shift = a_shift;
        prm.b_shift = b_shift;

        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ln.grid), 1, 1);
        cfg.blockDim = dim3(ln.k.threads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(ln.k.smem_bytes);
        cfg.stream = static_cast<cudaStream_t>(stream);
        cfg.numAttrs = 0;
        void* args4[4] = {res ? static_cast<void*>(&resA) : &tmA, res ? static_cast<void*>(&resB) : &tmB, &tmB2,
                          &prm};
        void* args3[3] = {&tmA, &tmB, &prm};  // (the direct-A kernel takes no second B map)
        if (cudaLaunchKernelExC(&cfg, ln.k.fn, variant == 2 ? args3 : args4) != cudaSuccess) {
            (void)cudaGetLastError();
            rc = SGEMM_ERR_CUDA;
        }
    }
    if (ws_split) (void)cudaFreeAsync(ws_split, cs);
    if (ws) (void)cudaFreeAsync(ws, cs);
    packed.release();
    return rc;
}

}  // namespace detail
}  // namespace gb300
