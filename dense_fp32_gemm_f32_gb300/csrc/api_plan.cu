// Argument checks and the choice of FFMA variant (producer, tile, stages,
// schedule, repacking), tensor-map encoding, and the variant's name.
#include "api_internal.h"

namespace gb300 {
namespace detail {

bool ranges_overlap(const void* a, size_t abytes, const void* b, size_t bbytes) {
    if (!abytes || !bbytes) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

size_t span_bytes(long long rows, long long cols, long long ld) {
    if (rows <= 0 || cols <= 0) return 0;
    return static_cast<size_t>(((rows - 1) * ld + cols) * 4);
}

// a_mn: A is stored transposed (K x M, lda >= M); b_nk: B is stored
// transposed (N x K, ldb >= K).
int validate(int M, int N, int K, const float* A, int lda, const float* B, int ldb, const float* C, int ldc,
             bool a_mn, bool b_nk) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (lda < (a_mn ? M : K) || ldb < (b_nk ? K : N) || ldc < N) return SGEMM_ERR_INVALID_ARG;
    if (M > 0 && K > 0 && !A) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && N > 0 && !B) return SGEMM_ERR_INVALID_ARG;
    if (M > 0 && N > 0 && !C) return SGEMM_ERR_INVALID_ARG;
    // Every operand is an array of floats: 4-byte aligned.
    if (((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 3u) != 0)
        return SGEMM_ERR_INVALID_ARG;
    // Output tiles are numbered with a 32-bit int.
    if (((static_cast<long long>(M) + kBM - 1) / kBM) * (((static_cast<long long>(N) + kBN - 1) / kBN) + 1) >
        0x7fffffffLL)
        return SGEMM_ERR_INVALID_ARG;
    const size_t cb = span_bytes(M, N, ldc);
    if (ranges_overlap(C, cb, A, a_mn ? span_bytes(K, M, lda) : span_bytes(M, K, lda)) ||
        ranges_overlap(C, cb, B, b_nk ? span_bytes(N, K, ldb) : span_bytes(K, N, ldb)))
        return SGEMM_ERR_INVALID_ARG;
    return SGEMM_OK;
}

// A read in the transposed layout: the consumers read each k's A values as
// two 16-byte vectors instead of a 4-k vector per row (82 -> 89 % FMA-pipe
// duty).  Two ways to get there: a transposing copy of A in HBM
// (sgemm_options.a_layout = 2; the transposed-A kernels, no extra work in
// the kernel) or two producer warps transposing each A slice in shared
// memory (SGEMM_PRODUCER_TMA_X; no copy, a little more shared-memory traffic
// in the kernel).  Measured on GB300 (TFLOP/s, A read as stored / copy in HBM
// / transposed in shared memory): 2048^3 62.0 / 62.7 / 66.9, 4096^3 65.4 /
// 68.5 / 70.5, 8192^3 66.4 / 71.2 / 71.0, 128 x 8192 x 16384 64.2 / 68.2 /
// 68.7, 8192 x 128 x 8192 62.0 / - / 66.4.  The copy costs one read and one
// write of A (~1/N of the product) and a pool buffer of A's size; with the
// two transposing warps it no longer wins anywhere, so it is taken only when
// forced (a_layout = 2) and the transposition in shared memory is automatic
// (make_plan).  (The general entry's A stored transposed is read in place by
// the transposed-A kernels: no copy.)

bool options_force_variant(const sgemm_options* opt) {
    return opt && (opt->producer || opt->split_k || opt->multicast || opt->math || opt->stages || opt->tail_split ||
                   opt->stream_k || opt->tile_n || opt->repack || opt->group_m || opt->l2_hint || opt->tile_k ||
                   opt->edge);
}

// 0 = keep A as stored, 1 = copy it transposed; -1 = invalid option.
int choose_a_layout(int K, const sgemm_options* opt) {
    const int want = opt ? opt->a_layout : 0;
    if (want < 0 || want > 2) return -1;
    return (K > 0 && want == 2) ? 1 : 0;
}



bool is_tma(int producer) {
    return producer == kProducerTma || producer == kProducerTmaWg || producer == kProducerFused ||
           producer == kProducerTmaX;
}

KernelEntry ffma_kernel(const Plan& pl) {
    if (pl.a_mn) return pl.producer == kProducerTma     ? ffma_kernel_amn(pl.stages, pl.math, false)
                        : pl.producer == kProducerTmaWg ? ffma_kernel_tma_wide_amn(pl.stages, pl.math)
                                                        : KernelEntry{nullptr, 0, 0};
    if (pl.producer == kProducerFused) return ffma_kernel_tma_fused(pl.stages, pl.math);
    if (pl.producer == kProducerLdg) return ffma_kernel_ldg(pl.stages, pl.math);
    if (pl.res)
        return pl.producer == kProducerTmaX ? ffma_kernel_res(pl.stages, pl.math, false, pl.ec > 0)
                                            : KernelEntry{nullptr, 0, 0};
    if (pl.producer == kProducerTmaX)
        return pl.bk == kBK16 ? ffma_kernel_tma_x16(pl.stages, pl.math)
                              : ffma_kernel_tma_x(pl.stages, pl.math, false, pl.ec > 0);
    if (pl.bn == kBNWide) return pl.producer == kProducerTmaWg ? ffma_kernel_tma_wide(pl.stages, pl.math)
                                                                : KernelEntry{nullptr, 0, 0};
    switch (pl.producer) {
        case kProducerTma: return ffma_kernel_tma(pl.stages, pl.math);
        case kProducerTmaWg: return ffma_kernel_tma_wg(pl.stages, pl.math);
        case kProducerCpAsync: return ffma_kernel_cpasync(pl.stages, pl.math);
    }
    return {nullptr, 0, 0};
}

const char* producer_name(int producer) {
    switch (producer) {
        case kProducerTma: return "tma";
        case kProducerTmaWg: return "tmawg";
        case kProducerFused: return "fused";
        case kProducerTmaX: return "tmax";
        case kProducerCpAsync: return "cpasync";
        case kProducerLdg: return "ldg";
    }
    return "?";
}

bool tma_ok(const float* p, int ld) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (static_cast<long long>(ld) * 4) % 16 == 0;
}

// Chooses the variant.  Any field of `opt` that is non-zero forces that choice.
int make_plan(const DeviceState& st, int M, int N, int K, const float* A, int lda, const float* B, int ldb,
              const sgemm_options* opt, Plan* out, bool a_mn, bool b_nk, bool scaled) {
    Plan pl;
    // B stored N x K (general entry only): tensor-map readable B, 128 x 128
    // tiles, 2 stages, paired FMA, and a transposing warp for B.
    if (b_nk && (K == 0 || !tma_ok(B, ldb) || (opt && options_force_variant(opt))))
        return SGEMM_ERR_INVALID_ARG;
    pl.b_nk = b_nk;
    // Cluster multicast of the operand slices is not built (see the
    // multicast field of sgemm_options).
    if (opt && (opt->multicast < 0 || opt->multicast > 2)) return SGEMM_ERR_INVALID_ARG;
    if (opt && opt->multicast == 2) return SGEMM_ERR_NOT_IMPLEMENTED;
    // Transposed A (general entry only): tensor-map readable A, TMA producer
    // warp, 2 stages, paired FMA.
    if (a_mn && (K == 0 || !tma_ok(A, lda) ||
                 (opt && (opt->producer || (opt->tile_n && opt->tile_n != kBNWide) || opt->math || opt->stages))))
        return SGEMM_ERR_INVALID_ARG;
    pl.a_mn = a_mn;
    // K slice depth: 32, or 16 when forced (the transposing producer only).
    const int want_bk = opt ? opt->tile_k : 0;
    if (want_bk != 0 && want_bk != kBK && want_bk != kBK16) return SGEMM_ERR_INVALID_ARG;
    pl.bk = want_bk == kBK16 ? kBK16 : kBK;
    if (pl.bk == kBK16 && (a_mn || b_nk)) return SGEMM_ERR_INVALID_ARG;
    pl.num_k_tiles = static_cast<int>(ceil_div(K, pl.bk));
    long long tiles_n = ceil_div(N, kBN);
    const long long tiles_m = ceil_div(M, kBM);

    // Producer: tensor maps need 16-byte aligned bases and row strides, and
    // K > 0.  An operand without them is either repacked into pitched rows
    // (which the tensor maps can address) or read by the cp.async producer;
    // the loader warps (kProducerLdg) read any alignment too, but only when
    // forced: measured on GB300 they run at 19-25 TFLOP/s on 1023 x 1025 x
    // 1027 ... 8191 x 8193 x 8195 with 2, 3 or 4 stages alike, against 35-67
    // repacked and 32-50 with cp.async (each slice's row loads cost them a
    // memory round trip that the consumers' 2 us per slice does not cover).
    const int want_prod = opt ? opt->producer : 0;
    const int want_repack = opt ? opt->repack : 0;
    if (want_repack < 0 || want_repack > 2) return SGEMM_ERR_INVALID_ARG;
    const int misaligned = (a_mn || tma_ok(A, lda) ? 0 : 1) | (tma_ok(B, ldb) ? 0 : 2);
    // Residue-class tensor maps (operands of any alignment read in place):
    // every class of rows mod 4 must hold a row of A and of B (M, K >= 4);
    // the kernels have 128 x 128 tiles, 32-deep slices and paired FMA, with
    // the plain epilogue on 2 to 4 stages and the scaled one on 2.
    // Automatic for misaligned operands below kResMaxFlops, and whenever
    // copies are ruled out (repack = 1).
    const double flops = 2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K);
    const bool res_ok = !a_mn && !b_nk && M >= 4 && K >= 4 && !(scaled && opt && opt->stages && opt->stages != 2) &&
                        !(opt && opt->tile_n && opt->tile_n != kBN) &&
                        !(opt && opt->tile_k && opt->tile_k != kBK) &&
                        !(opt && opt->stages && (opt->stages < 2 || opt->stages > 4)) &&
                        !(opt && opt->math && opt->math != kMathFfma2);
    if (want_prod == SGEMM_PRODUCER_TMA_RES) {
        if (!res_ok || want_repack == 2) return SGEMM_ERR_INVALID_ARG;
        pl.res = true;
    } else if (want_prod == SGEMM_PRODUCER_AUTO && misaligned && res_ok &&
               (want_repack == 1 || (want_repack == 0 && flops < kResMaxFlops))) {
        pl.res = true;
    }
    if (!pl.res && K > 0 && misaligned &&
        (want_repack == 2 || a_mn || b_nk ||  // (the transposed-operand kernels have no cp.async form)
         (want_repack == 0 && want_prod == SGEMM_PRODUCER_AUTO && flops >= kRepackMinFlops)))
        pl.repack = misaligned;
    const bool aligned = K > 0 && (misaligned & ~pl.repack) == 0;
    if (pl.res) {
        pl.producer = kProducerTmaX;
    } else if (want_prod == SGEMM_PRODUCER_TMA) {
        if (!aligned) return SGEMM_ERR_INVALID_ARG;
        pl.producer = kProducerTma;
    } else if (want_prod == SGEMM_PRODUCER_TMA_WG) {
        if (!aligned) return SGEMM_ERR_INVALID_ARG;
        if (!st.regsplit_ok) return SGEMM_ERR_UNSUPPORTED;
        pl.producer = kProducerTmaWg;
    } else if (want_prod == SGEMM_PRODUCER_TMA_X) {
        if (!aligned || a_mn) return SGEMM_ERR_INVALID_ARG;
        pl.producer = kProducerTmaX;
    } else if (want_prod == SGEMM_PRODUCER_FUSED) {
        if (!aligned) return SGEMM_ERR_INVALID_ARG;
        pl.producer = kProducerFused;
    } else if (want_prod == SGEMM_PRODUCER_CPASYNC) {
        pl.producer = kProducerCpAsync;
    } else if (want_prod == SGEMM_PRODUCER_LDG) {
        if (K == 0 || a_mn || b_nk) return SGEMM_ERR_INVALID_ARG;
        pl.producer = kProducerLdg;
    } else if (want_prod == SGEMM_PRODUCER_AUTO) {
        // Tensor maps: A transposed in shared memory, unless it already is in
        // HBM (a_mn) or another choice rules the transposing warps out.
        const int max_x_stages = (opt && opt->tile_k == kBK16) ? 6 : 4;
        const bool x_ok = !a_mn && !(opt && ((opt->tile_n && opt->tile_n != kBN) ||
                                             (opt->stages && (opt->stages < 2 || opt->stages > max_x_stages))));
        // (b_nk: B is aligned, checked above; A is aligned or repacked.)
        pl.producer = !aligned ? kProducerCpAsync : x_ok ? kProducerTmaX : kProducerTma;
    } else {
        return SGEMM_ERR_INVALID_ARG;
    }

    // Tile width: 128 x 256 tiles need the producer warpgroup (register
    // split) and so tensor maps.
    const int want_bn = opt ? opt->tile_n : 0;
    if (want_bn == kBNWide) {
        if (want_prod == SGEMM_PRODUCER_AUTO) {
            if (!aligned) return SGEMM_ERR_INVALID_ARG;
            if (!st.regsplit_ok) return SGEMM_ERR_UNSUPPORTED;
            pl.producer = kProducerTmaWg;
        }
        if (pl.producer != kProducerTmaWg) return SGEMM_ERR_INVALID_ARG;
        pl.bn = kBNWide;
    } else if (want_bn == kBNFused) {
        // 128 x 64 tiles: the fused-producer CTAs, two per SM.
        if (want_prod == SGEMM_PRODUCER_AUTO) {
            if (!aligned) return SGEMM_ERR_INVALID_ARG;
            pl.producer = kProducerFused;
        }
        if (pl.producer != kProducerFused) return SGEMM_ERR_INVALID_ARG;
    } else if (want_bn != 0 && want_bn != kBN) {
        return SGEMM_ERR_INVALID_ARG;
    }
    if (pl.producer == kProducerFused) pl.bn = kBNFused;

    if (opt && opt->math) {
        if (opt->math != kMathFfma && opt->math != kMathFfma2) return SGEMM_ERR_INVALID_ARG;
        pl.math = opt->math;
    }
    // Stages: two for the tensor-map producers (measured on GB300 with the
    // paired-FMA consumers: 0.3-2 % faster than 3-6 at every named problem,
    // 20-25 % faster than one), four for cp.async, whose 4-byte copies have
    // more latency to hide.
    pl.stages = pl.producer == kProducerCpAsync ? 4 : pl.producer == kProducerLdg ? 3 : 2;
    if (opt && opt->stages) {
        if (opt->stages < 1 || opt->stages > 6) return SGEMM_ERR_INVALID_ARG;
        pl.stages = opt->stages;
    }
    if (pl.producer == kProducerCpAsync && pl.stages != 2 && pl.stages != 4) {
        if (opt && opt->stages) return SGEMM_ERR_INVALID_ARG;
        pl.stages = 4;
    }
    if (pl.producer == kProducerFused && !(opt && opt->stages)) pl.stages = 4;
    // (16-deep slices: 4 stages by default, the same 64 k of lookahead as two
    // 32-deep ones; up to 6.)
    if (pl.bk == kBK16 && !(opt && opt->stages)) pl.stages = 4;
    if ((pl.bn == kBNWide || pl.bn == kBNFused || pl.producer == kProducerTmaX) &&
        (pl.stages < 2 || pl.stages > (pl.producer == kProducerTmaX && pl.bk == kBK16 ? 6 : 4)))
        return SGEMM_ERR_INVALID_ARG;
    if (pl.producer == kProducerTmaX && pl.bn != kBN) return SGEMM_ERR_INVALID_ARG;
    if (pl.res && (pl.stages > (scaled ? 2 : 4) || pl.math != kMathFfma2 || pl.bk != kBK))
        return SGEMM_ERR_INVALID_ARG;
    if (pl.producer == kProducerLdg && (pl.bn != kBN || pl.bk != kBK || pl.stages < 2 || pl.stages > 4))
        return SGEMM_ERR_INVALID_ARG;
    if (pl.bk == kBK16 && (pl.producer != kProducerTmaX || pl.stages == 5)) return SGEMM_ERR_INVALID_ARG;
    // CTAs that can be resident at once, for the stream-K grid.
    const int per_sm = pl.producer == kProducerFused ? st.fused_per_sm[pl.stages] : 1;
    if (per_sm < 1) return SGEMM_ERR_UNSUPPORTED;
    const long long slots = static_cast<long long>(st.sm_count) * per_sm;

    // Stream-K (decided first; see below for the schedule).  Automatic
    // whenever nothing else is forced and there are at least two (tile, K
    // slice) units per SM: measured on GB300 it beats the plain grid and
    // cluster split-K (1024^3 +8 %, 2048^3 +16 %, 4096^3 +4 %, 8192^3 +1 %,
    // 8192x128x8192 +22 %); tiny problems keep cluster split-K.
    const int want_sk = opt ? opt->stream_k : 0;
    if (want_sk < 0 || want_sk > 2) return SGEMM_ERR_INVALID_ARG;
    const bool forced_other = opt && (opt->split_k || opt->tail_split > 1);
    auto stream_k_for = [&](long long tiles) {
        return want_sk == 2 ||
               (want_sk == 0 && !forced_other && pl.num_k_tiles > 0 && tiles * pl.num_k_tiles >= 2LL * slots);
    };

    // Thin column edge (sgemm_options.edge): when N mod 128 is 1 to
    // kEdgeMaxCols, the stream-K launches of the transposing producer with
    // the plain epilogue compute those columns with the last column of full
    // tiles (FfmaParams ec) instead of giving them a column of tiles of their
    // own, whose units would cost as much as full ones: 1023 x 1025 x 1027
    // has 64 tiles of 33 K slices instead of 72 (14 units on the busiest SM
    // instead of 16).
    const int want_edge = opt ? opt->edge : 0;
    if (want_edge < 0 || want_edge > 1) return SGEMM_ERR_INVALID_ARG;
    const int ec = static_cast<int>(N % kBN);
    const bool edge_ok = want_edge == 0 && pl.producer == kProducerTmaX && pl.bn == kBN && pl.bk == kBK &&
                         pl.math == kMathFfma2 && !scaled && !a_mn && !b_nk && ec >= 1 && ec <= kEdgeMaxCols &&
                         N > kBN &&
                         stream_k_for((N / kBN) * tiles_m);
    tiles_n = edge_ok ? N / kBN : ceil_div(N, pl.bn);
    const long long tiles = tiles_n * tiles_m;
    const bool use_sk = stream_k_for(tiles);
    pl.ec = edge_ok ? ec : 0;

    // Split-K over the whole grid, only when the tiles do not fill one wave:
    // pick s in 1..8 minimising (waves of clusters) x (K tiles per CTA).  (With
    // a wave or more, only the last partial wave is split; see below.)
    int split = 1;
    if (opt && opt->split_k) {
        if (opt->split_k < 1 || opt->split_k > 8) return SGEMM_ERR_INVALID_ARG;
        split = opt->split_k;
    } else if (tiles < st.sm_count && !use_sk && pl.producer != kProducerFused) {
        long long best = -1;
        for (int s = 1; s <= 8; ++s) {
            const int slots = st.max_clusters_split[s];
            if (slots <= 0) continue;
            if (s > 1 && pl.num_k_tiles < 2 * s) break;  // keep at least two K slices per CTA
            const long long cost = ceil_div(tiles, slots) * ceil_div(pl.num_k_tiles, s);
            if (best < 0 || cost < best) {
                best = cost;
                split = s;
            }
        }
    }
    if (split > 1 && pl.stages < 2) return SGEMM_ERR_INVALID_ARG;  // partial tile needs 64 KiB of ring
    if (split > 1 && pl.producer == kProducerFused) return SGEMM_ERR_INVALID_ARG;  // two CTAs per SM: no clusters

    pl.tiles_n = static_cast<int>(tiles_n);
    pl.tiles_m = static_cast<int>(tiles_m);
    const long long grid_tiles = static_cast<long long>(pl.tiles_n) * tiles_m;

    // Tile order (see tile_rc): groups of rows of tiles, walked column by
    // column (odd groups from the right), so that a wave of 152 CTAs covers
    // about 16 x 9.5 tiles at 4096^3.  Row by row, a wave of the 4096^3
    // product needs ~5 A row panels and all 32 B column panels, and B is read
    // from HBM once per wave.  Measured with ncu on GB300 (DRAM bytes read
    // per launch; A and B hold 134 MB at 4096^3, 537 MB at 8192^3): 4096^3
    // 533 MB row by row, 376 / 290 / 556 MB in groups of 8 / 16 / 32 rows,
    // 276 MB in groups of 16 walked alternately; 8192^3 8.3 GB row by row,
    // 3.4 / 3.7 GB in groups of 8 / 16 walked alternately.  The time does
    // not change (the kernel is bound by the FP32 pipe, HBM ~4 % busy).  The
    // group holds as many rows as keep its A panels within kGroupABytes.
    const int want_group = opt ? opt->group_m : 0;
    if (want_group < 0) return SGEMM_ERR_INVALID_ARG;
    const long long panel = static_cast<long long>(kBM) * (K > 0 ? K : 1) * 4;
    const long long auto_group = std::max<long long>(kGroupRowsMin, std::min<long long>(kGroupRowsMax, kGroupABytes / panel));
    pl.group_m = want_group > 0 ? want_group : static_cast<int>(auto_group);
    if (pl.group_m > pl.tiles_m) pl.group_m = pl.tiles_m > 0 ? pl.tiles_m : 1;
    const int want_hint = opt ? opt->l2_hint : 0;
    if (want_hint < 0 || want_hint > 4) return SGEMM_ERR_INVALID_ARG;
    pl.a_evict_last = (want_hint == 2 || want_hint == 3) ? 1 : 0;
    pl.b_evict_first = want_hint == 3 ? 1 : 0;
    // C's tensor-map stores (K >= 4096 slices; see kTmaStoreMinSlices) carry
    // the evict-first policy by default, so that C streaming through L2 does
    // not push out the A and B panels the next tiles read: measured with ncu
    // at 4096^3, 323 MB of DRAM traffic per launch against 337 MB without a
    // policy and 329 MB with A's slices evict-last, the time unchanged.
    pl.c_evict_first = (want_hint == 0 || want_hint == 4) ? 1 : 0;

    // Last partial wave.  When the tiles do not fill a whole number of waves,
    // the last wave leaves SMs idle for a full tile time.  Those tiles can run
    // as a second launch split along K (clusters + shared-memory reduction),
    // so that more CTAs share the tail at 1/s of the work each; the modelled
    // tail time, in full-K tile times, is ceil(rem / clusters_s) / s.  On
    // GB300 the measured tail is well above that model (4096^3: 112 tail tiles
    // split 5 ways made the call 3 % slower; 2048^3: 104 tiles split 4 ways,
    // 2.6 % faster), so it is taken only when forced (tail_split = 2..8).
    pl.nlaunch = 1;
    pl.launch[0].tile_base = 0;
    pl.launch[0].tiles = static_cast<int>(grid_tiles);
    pl.launch[0].split = split;
    const int want_tail = opt ? opt->tail_split : 0;
    if (want_tail < 0 || want_tail > 8) return SGEMM_ERR_INVALID_ARG;
    if (split == 1 && want_tail > 1 && grid_tiles > st.sm_count && pl.producer != kProducerFused) {
        const long long full = (grid_tiles / st.sm_count) * st.sm_count;
        const long long rem = grid_tiles - full;
        // keep at least four K slices per CTA of the tail
        if (rem > 0 && st.max_clusters_split[want_tail] > 0 && pl.num_k_tiles >= 4 * want_tail) {
            pl.nlaunch = 2;
            pl.launch[0].tiles = static_cast<int>(full);
            pl.launch[1].tile_base = static_cast<int>(full);
            pl.launch[1].tiles = static_cast<int>(rem);
            pl.launch[1].split = want_tail;
        }
    }

    // Stream-K schedule: one CTA per SM (two for the fused producer), partial
    // tiles finished through a global workspace.
    if (use_sk) {
        if (split > 1 || pl.nlaunch > 1 || pl.num_k_tiles == 0) return SGEMM_ERR_INVALID_ARG;
        // All but the last full wave run data-parallel (raster order keeps
        // the A and B panels in flight few, as in the plain launch); the last
        // full wave and the partial one are dealt out as units.
        const long long G = slots;
        const long long waves = grid_tiles / G;
        const long long dp = waves > 1 ? (waves - 1) * G : 0;
        const long long units = (grid_tiles - dp) * pl.num_k_tiles;
        pl.sk = 1;
        pl.sk_dp_tiles = static_cast<int>(dp);
        pl.nlaunch = 1;
        pl.launch[0].tile_base = 0;
        pl.launch[0].split = 1;
        pl.launch[0].tiles = static_cast<int>(units < G ? units : G);
    }
    *out = pl;
    return SGEMM_OK;
}

int encode_2d(CUtensorMap* map, const float* base, long long inner, long long outer, long long ld, int box_inner,
              int box_outer, CUtensorMapSwizzle swz) {
    if (!g_encode) return SGEMM_ERR_UNSUPPORTED;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGEMM_OK : SGEMM_ERR_CUDA;
}

// The four residue-class maps of a rows x cols operand with pitch ld (rows
// >= 4, so that every class holds a row): class j holds rows j, j + 4,
// ..., (rows - j + 3) / 4 of them, 4 ld floats apart; its map is based at the
// 16-byte block boundary at or before row j's first element, t_j floats
// before it, and spans cols + t_j floats per row, so that the row's last
// element is the last inside the map.  shifts gets t_j in bits 2j, 2j + 1.
// Boxes of box_inner x box_outer, no swizzle.
int encode_res(ResMaps* maps, int* shifts, const float* base, long long rows, long long cols, long long ld,
               int box_inner, int box_outer) {
    if (rows < 4) return SGEMM_ERR_INVALID_ARG;
    int sh = 0;
    for (int j = 0; j < 4; ++j) {
        const uintptr_t start = reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>(j) * ld * 4;
        const int t = static_cast<int>((start & 15u) >> 2);
        const float* b = reinterpret_cast<const float*>(start - (start & 15u));
        const int rc = encode_2d(&maps->m[j], b, cols + t, (rows - j + 3) / 4, 4 * ld, box_inner, box_outer,
                                 CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != SGEMM_OK) return rc;
        sh |= t << (2 * j);
    }
    *shifts = sh;
    return SGEMM_OK;
}

const char* describe_plan(const Plan& pl) {
    static thread_local char buf[128];
    int n = std::snprintf(buf, sizeof buf, "%s/%s/s%d/st%d", producer_name(pl.producer),
                          pl.math == kMathFfma2 ? "ffma2" : "ffma", pl.launch[0].split, pl.stages);
    if (pl.nlaunch > 1 && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/tail%d:%d", pl.launch[1].split, pl.launch[1].tiles);
    if (pl.sk && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/sk%d", pl.launch[0].tiles);
    if (pl.bn != kBN && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/n%d", pl.bn);
    if (pl.repack && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/repack%s", pl.repack == 1 ? "A" : pl.repack == 2 ? "B" : "AB");
    if (pl.a_mn && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/at");
    if (pl.b_nk && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/bt");
    if (pl.bk != kBK && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/k%d", pl.bk);
    if (pl.res && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/res");
    if (pl.ec && n > 0 && n < static_cast<int>(sizeof buf))
        std::snprintf(buf + n, sizeof buf - n, "/ec%d", pl.ec);
    return buf;
}


// Small problems: the 32 x 32-tile kernel when the 128 x 128 tiles would be
// too few to occupy the GPU and the product is small (see small_problem).
constexpr double kSmallMaxFlops = 268435456.0;  // 2^28

bool small_problem(const DeviceState& st, int M, int N, int K) {
    const long long tiles = ceil_div(M, kBM) * ceil_div(N, kBN);
    return 2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) <= kSmallMaxFlops &&
           4 * tiles <= st.sm_count;
}

// A forced small kernel takes no other forced choice (it has no producer,
// stages, split or tile options, and no waits for debug_skip_stage to time out).
bool small_forced_ok(const sgemm_options* opt) {
    return !(opt->split_k || opt->multicast || opt->math || opt->stages || opt->tail_split || opt->stream_k ||
             opt->group_m || opt->l2_hint || opt->tile_k ||
             opt->tile_n || opt->repack || opt->a_layout || opt->debug_skip_stage);
}

}  // namespace detail
}  // namespace gb300
