// FP32 matrix multiply on the fifth-generation tensor cores (tcgen05), sm_103a,
// with the three-product TF32 split.
//
// C (M x N) = A (M x K) * B (K x N), all row-major float32.
//
// Tensor cores have no FP32 multiply-add, but they multiply TF32 values (10
// explicit mantissa bits) exactly and accumulate in FP32.  Each operand is
// split into a TF32 "big" part and the TF32 rounding of what is left:
//     a = a_big + a_small + e_a,  a_big = tf32(a),  a_small = tf32(a - a_big),
// with |e_a| <= 2^-22 |a|, and the product is taken as
//     a*b ~ a_small*b_big + a_big*b_small + a_big*b_big,
// dropping a_small*b_small and the e terms, each below 2^-22 |a||b|: about
// 1e-6 of sum_k |a||b| in all, far inside the 5e-5 contract.  Integers in
// {-8..8} are exact in TF32, so their small parts are 0 and the result is
// exact.  (The pages mention tensor cores only as a future direction of the
// "Hardware acceleration" page's summary; nothing of this is on the pages.)
//
// One CTA computes a 128 x BN tile of C (TcShape<BN, BK>: 128 x 128 with
// K-slices of 32 and 128-byte operand rows, or 128 x 256 with K-slices of 16
// and 64-byte rows); 10 warps:
//   warp 0      TMA producer: A and B K-slices into the raw stages;
//   warp 1      allocates BN tensor-memory columns (the FP32 accumulator)
//               and one lane issues the MMAs: per K-slice BK / 8 k-steps of
//               8, three tcgen05.mma.kind::tf32 each (small*big, big*small,
//               big*big), then tcgen05.commit releases the split stage;
//   warps 2..9  split the raw K-slice into four K-major, swizzled TF32
//               operand tiles (A_big, A_small, B_big, B_small) in 2 split
//               stages (B is transposed on the way: it arrives with n
//               innermost), then, after the last MMA, read the accumulator
//               out of tensor memory (tcgen05.ld) and store C.  Eight warps
//               (two per SM sub-partition) so that one warp's shared-memory
//               latency hides behind the other's conversions.
//
// Every wait is bounded by `timeout_ns`; on expiry the thread records the
// timeout in the status word, stops working, and still reaches the final CTA
// barrier, after which warp 1 frees the tensor memory.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "sgemm_3xtf32_params.h"

namespace gb300 {

__device__ __forceinline__ void split_tf32(float x, float& big, float& small) {
    big = to_tf32_rna(x);
    small = to_tf32_rna(x - big);  // x - big is exact in FP32
}

// K-major operand descriptor for the shape's swizzle (128- or 64-byte rows).
template <int BK>
__device__ __forceinline__ uint64_t tc_operand_desc(uint32_t saddr) {
    if constexpr (BK == 32)
        return umma_desc_kmajor_sw128(saddr);
    else
        return umma_desc_kmajor_sw64(saddr);
}

// The last CTA of a K-split tile: C[tile] = ((C + P_1) + P_2) + ... over the
// later parts' partial tiles P_q in ws, element by element in part order (C
// holds part 0's result).  Elements beyond M or N are not touched.  One SM
// does this alone, so it is bound by the latency of its loads: each thread
// takes 13 groups of 4 columns (g, g + 320, ...; a whole 128 x 128 tile in
// one pass) and issues all their loads before any add or store.  L2 reads
// (__ldcg), since other SMs wrote these lines during this launch.
template <int BN>
__device__ __forceinline__ void tc_split_finish(const TcParams& p, int local, int ks, int m0, int n0) {
    constexpr int kBM = kTcBM;
    constexpr int kGroups = kBM * BN / 4;
    constexpr int kPer = (kTcBM * kTcBN / 4 + kTcThreads - 1) / kTcThreads;
    const int rows = min(kBM, p.M - m0), cols = min(BN, p.N - n0);
    const long long part_floats = static_cast<long long>(kBM) * BN;
    const float* const w = p.ws + static_cast<long long>(local) * (ks - 1) * part_floats;
    for (int g0 = static_cast<int>(threadIdx.x); g0 < kGroups; g0 += kPer * kTcThreads) {
        float4 a[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int g = g0 + j * kTcThreads;
            const int r = g / (BN / 4), c = 4 * (g % (BN / 4));
            const bool row_in = g < kGroups && r < rows;
            const float* out = p.C + static_cast<long long>(m0 + r) * p.ldc + n0 + c;
            if (p.vec_store && row_in && c + 3 < cols) {
                a[j] = __ldcg(reinterpret_cast<const float4*>(out));
            } else {
                a[j].x = row_in && c < cols ? __ldcg(out) : 0.f;
                a[j].y = row_in && c + 1 < cols ? __ldcg(out + 1) : 0.f;
                a[j].z = row_in && c + 2 < cols ? __ldcg(out + 2) : 0.f;
                a[j].w = row_in && c + 3 < cols ? __ldcg(out + 3) : 0.f;
            }
        }
        for (int q = 0; q < ks - 1; ++q) {
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int g = g0 + j * kTcThreads;
                if (g < kGroups) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(
                        w + q * part_floats + static_cast<long long>(g / (BN / 4)) * BN + 4 * (g % (BN / 4))));
                    a[j].x += v.x;
                    a[j].y += v.y;
                    a[j].z += v.z;
                    a[j].w += v.w;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int g = g0 + j * kTcThreads;
            const int r = g / (BN / 4), c = 4 * (g % (BN / 4));
            if (g >= kGroups || r >= rows) continue;
            float* out = p.C + static_cast<long long>(m0 + r) * p.ldc + n0 + c;
            if (p.vec_store && c + 3 < cols) {
                *reinterpret_cast<float4*>(out) = a[j];
            } else {
                if (c < cols) out[0] = a[j].x;
                if (c + 1 < cols) out[1] = a[j].y;
                if (c + 2 < cols) out[2] = a[j].z;
                if (c + 3 < cols) out[3] = a[j].w;
            }
        }
    }
}

// PB: B's TF32 parts come pre-split and transposed (N x K) from HBM: tmB maps
// the big part and tmB2 the small part, each loaded by the TMA into its slot
// of the split stage (arriving on split_full with the split warps, which then
// write A's parts only).  Without PB, tmB maps B as stored and tmB2 is unused.
//
// RES: A and B of any alignment, read in place through residue-class maps
// (tmA and tmB are four maps each; res_maps.cuh): the split warps take A's
// 16-byte chunk (row m, k = 4c..4c+3) as the two aligned vectors of its class
// box row that hold it, shifted by the class's t, and B's elements from their
// class box rows at t + n.
template <int BN, int BK, bool PB = false, bool RES = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    sgemm_3xtf32_kernel(const __grid_constant__ MapsFor<RES> tmA, const __grid_constant__ MapsFor<RES> tmB,
                        const __grid_constant__ CUtensorMap tmB2, const TcParams p) {
    using T = TcShape<BN, BK, PB, RES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    auto rawA = [&](int r) { return base + static_cast<uint32_t>(r * T::kRawABytes); };
    auto rawB = [&](int r) { return base + static_cast<uint32_t>(T::kRawStages * T::kRawABytes + r * T::kRawBBytes); };
    auto split = [&](int s) {
        return base + static_cast<uint32_t>(T::kRawStages * (T::kRawABytes + T::kRawBBytes) + s * T::kSplitBytes);
    };
    const uint32_t bars = base + T::kRingBytes;
    constexpr uint32_t R = T::kRawStages, S = T::kSplitStages;
    auto raw_full = [&](int r) { return bars + 8u * r; };
    auto raw_empty = [&](int r) { return bars + 8u * (R + r); };
    auto split_full = [&](int s) { return bars + 8u * (2 * R + s); };
    auto split_empty = [&](int s) { return bars + 8u * (2 * R + S + s); };
    const uint32_t acc_full = bars + 8u * (2 * R + 2 * S);
    const uint32_t tmem_slot = acc_full + 8u;
    int* const last_part = reinterpret_cast<int*>(smem_raw + (tmem_slot + 4u - raw_base));  // K split
    static_assert(8 * (2 * T::kRawStages + 2 * T::kSplitStages + 1) + 8 <= 256, "barrier area");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Tile and K range: the whole K for one tile per CTA, or (k_split = s) one
    // of s parts of it, CTAs s t .. s t + s - 1 sharing tile tile_base + t.
    // K slices are counted from kbase: nkt slices here.
    const int ks = p.k_split > 1 ? p.k_split : 1;
    const bool ksplit = ks > 1;
    const int local = static_cast<int>(blockIdx.x) / ks;  // this launch's tile index
    const int part = static_cast<int>(blockIdx.x) % ks;
    const int tile = p.tile_base + local;
    const int m0 = (tile / p.tiles_n) * T::kBM;
    const int n0 = (tile % p.tiles_n) * BN;
    const int kbase = (p.num_k_tiles * part) / ks;
    const int nkt = (p.num_k_tiles * (part + 1)) / ks - kbase;
    const bool second = part > 0;  // a later part: its partial tile goes to ws
    const unsigned long long tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int r = 0; r < T::kRawStages; ++r) {
            mbar_init(raw_full(r), 1);
            mbar_init(raw_empty(r), kTcSplitWarps);  // one arrival per split warp
        }
        for (int s = 0; s < T::kSplitStages; ++s) {
            mbar_init(split_full(s), kTcSplitWarps + (PB ? 1 : 0));  // (+ the producer, for B's parts)
            mbar_init(split_empty(s), 1);  // tcgen05.commit
        }
        mbar_init(acc_full, 1);
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, T::kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    if (warp == 0 && lane == 0) {
#pragma unroll
        for (int j = 0; j < (RES ? 4 : 1); ++j) {
            prefetch_tensormap(&res_map(tmA, j));
            prefetch_tensormap(&res_map(tmB, j));
        }
        if (PB) prefetch_tensormap(&tmB2);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    uint32_t tmem;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(tmem) : "r"(tmem_slot) : "memory");

    bool timed_out = false;
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued_round[T::kRawStages], issued_sround[T::kSplitStages];
#pragma unroll
            for (int r = 0; r < T::kRawStages; ++r) issued_round[r] = -1;
#pragma unroll
            for (int s = 0; s < T::kSplitStages; ++s) issued_sround[s] = -1;
            // (debug: the first CTA of the launch, with K split its first part)
            const bool skip_here = p.skip_stage > 0 && blockIdx.x == 0 && p.tile_base == 0;
            for (int kt = 0; kt < nkt; ++kt) {
                const int r = kt % T::kRawStages;
                const int round = kt / T::kRawStages;
                if (round > 0 && !mbar_wait_bounded(raw_empty(r), (round - 1) & 1, tmo)) {
                    timed_out = true;
                    break;
                }
                if (PB) {
                    // B's parts go straight into split stage s, once its MMAs are done.
                    const int s = kt % T::kSplitStages;
                    const int sround = kt / T::kSplitStages;
                    if (sround > 0 && !mbar_wait_bounded(split_empty(s), (sround - 1) & 1, tmo)) {
                        timed_out = true;
                        break;
                    }
                }
                if (skip_here && kt == p.skip_stage - 1) continue;
                const int kc = (kbase + kt) * BK;  // K coordinate of the slice
                mbar_arrive_expect_tx(raw_full(r), T::kRawABytes + T::kRawBBytes);
                if (RES) {
                    // Four class boxes per operand: A rows m0 / 4 .. + 31 of
                    // each class from kc, B rows kc / 4 .. + 7 from n0.
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        tma_load_2d(rawA(r) + j * kResAPlaneBytes, &res_map(tmA, j), raw_full(r), kc, m0 >> 2);
                        tma_load_2d(rawB(r) + j * kResBPlaneBytes, &res_map(tmB, j), raw_full(r), n0, kc >> 2);
                    }
                } else {
                    tma_load_2d(rawA(r), &tmA, raw_full(r), kc, m0);
                }
                if (PB) {
                    const int s = kt % T::kSplitStages;
                    const uint32_t b_big = split(s) + 2 * T::kOpABytes;
                    mbar_arrive_expect_tx(split_full(s), 2 * T::kOpBBytes);
                    tma_load_2d(b_big, &tmB, split_full(s), kc, n0);
                    tma_load_2d(b_big + T::kOpBBytes, &tmB2, split_full(s), kc, n0);
                    issued_sround[s] = kt / T::kSplitStages;
                } else if (!RES) {
                    tma_load_2d(rawB(r), &tmB, raw_full(r), n0, kc);
                }
                issued_round[r] = round;
            }
            for (int r = 0; r < T::kRawStages; ++r)  // drain: every issued copy has landed
                if (issued_round[r] >= 0 && !mbar_wait_bounded(raw_full(r), issued_round[r] & 1, tmo))
                    timed_out = true;
            if (PB) {
                // ... and B's parts: each split stage's last fill has completed
                // (its earlier fills completed before the MMAs freed it).
                for (int s = 0; s < T::kSplitStages; ++s)
                    if (issued_sround[s] >= 0 && !mbar_wait_bounded(split_full(s), issued_sround[s] & 1, tmo))
                        timed_out = true;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (int kt = 0; kt < nkt; ++kt) {
                const int s = kt % T::kSplitStages;
                if (!mbar_wait_bounded(split_full(s), (kt / T::kSplitStages) & 1, tmo)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_big = split(s), a_small = a_big + T::kOpABytes;
                const uint32_t b_big = a_big + 2 * T::kOpABytes, b_small = b_big + T::kOpBBytes;
#pragma unroll
                for (int kk = 0; kk < BK / 8; ++kk) {  // k-steps of 8 TF32 = 32 bytes of each row
                    const uint32_t off = static_cast<uint32_t>(kk * 32);
                    umma_tf32(tmem, tc_operand_desc<BK>(a_small + off), tc_operand_desc<BK>(b_big + off), T::kIdesc,
                              kt > 0 || kk > 0);
                    umma_tf32(tmem, tc_operand_desc<BK>(a_big + off), tc_operand_desc<BK>(b_small + off), T::kIdesc,
                              true);
                    umma_tf32(tmem, tc_operand_desc<BK>(a_big + off), tc_operand_desc<BK>(b_big + off), T::kIdesc,
                              true);
                }
                umma_commit(split_empty(s));  // stage s is free once these MMAs are done
            }
            umma_commit(acc_full);  // arrives when every MMA above has completed
            if (!mbar_wait_bounded(acc_full, 0, tmo)) timed_out = true;
        }
    } else {
        // ------------------------------------------------------------ split + epilogue
        const int tt = threadIdx.x - 64;  // 0 .. 32 * kTcSplitWarps - 1
        constexpr int kSplitThreads = 32 * kTcSplitWarps;
        constexpr int kAChunks = T::kRawABytes / 16 / kSplitThreads;  // 16-byte A chunks per thread
        constexpr int kBGroups = (BN * BK / 4) / kSplitThreads;  // (column, 4-k) groups per thread
        const int bn = tt % BN;                                      // B column of this thread
        const int bc0 = (tt / BN) * kBGroups;                        // its first 4-k group
        for (int kt = 0; kt < nkt; ++kt) {
            const int r = kt % T::kRawStages;
            const int s = kt % T::kSplitStages;
            if (!mbar_wait_bounded_warp(raw_full(r), (kt / T::kRawStages) & 1, tmo)) {
                timed_out = true;
                break;
            }
            // Loads are issued back to back before any use, so their latencies overlap.
            float4 av[kAChunks];
            if constexpr (RES) {
                // Chunk q of the swizzled K-major A tile: row m = q / 8, k =
                // 4c..4c+3 with c = (q mod 8) XOR (m mod 8).
                float4 v0[kAChunks], v1[kAChunks];
#pragma unroll
                for (int j = 0; j < kAChunks; ++j) {
                    const int q = tt + kSplitThreads * j;
                    const int m = q >> 3, c = (q & 7) ^ (m & 7);
                    const uint32_t src = rawA(r) + static_cast<uint32_t>((m & 3) * kResAPlaneBytes +
                                                                         (m >> 2) * (kResABox * 4) + c * 16);
                    v0[j] = lds128(src);
                    v1[j] = lds128(src + 16);
                }
#pragma unroll
                for (int j = 0; j < kAChunks; ++j) {
                    const int t = res_shift(p.a_shift, ((tt + kSplitThreads * j) >> 3) & 3);
                    av[j] = t == 0   ? v0[j]
                            : t == 1 ? make_float4(v0[j].y, v0[j].z, v0[j].w, v1[j].x)
                            : t == 2 ? make_float4(v0[j].z, v0[j].w, v1[j].x, v1[j].y)
                                     : make_float4(v0[j].w, v1[j].x, v1[j].y, v1[j].z);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kAChunks; ++j)
                    av[j] = lds128(rawA(r) + static_cast<uint32_t>((tt + kSplitThreads * j) * 16));
            }
            float bv[PB ? 1 : kBGroups][4];
            if constexpr (RES) {
                // k = 4 (bc0 + c) + i: class i, row bc0 + c of its box, at t_i + bn.
#pragma unroll
                for (int c = 0; c < kBGroups; ++c)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        asm volatile("ld.shared.f32 %0, [%1];"
                                     : "=f"(bv[c][i])
                                     : "r"(rawB(r) + static_cast<uint32_t>(i * kResBPlaneBytes +
                                                                           (bc0 + c) * (kResBBox * 4) +
                                                                           4 * (res_shift(p.b_shift, i) + bn))));
            } else if constexpr (!PB) {
                const uint32_t rb = rawB(r) + static_cast<uint32_t>(bn * 4);
#pragma unroll
                for (int c = 0; c < kBGroups; ++c)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        asm volatile("ld.shared.f32 %0, [%1];"
                                     : "=f"(bv[c][i])
                                     : "r"(rb + static_cast<uint32_t>((4 * (bc0 + c) + i) * BN * 4)));
            }
            if (kt >= T::kSplitStages &&
                !mbar_wait_bounded_warp(split_empty(s), ((kt / T::kSplitStages) - 1) & 1, tmo)) {
                timed_out = true;
                break;
            }
            const uint32_t a_big = split(s), a_small = a_big + T::kOpABytes;
            const uint32_t b_big = a_big + 2 * T::kOpABytes, b_small = b_big + T::kOpBBytes;
            // A: the TMA wrote the slice K-major with the same swizzle the MMA
            // reads, so the split is element-wise on 16-byte chunks.
#pragma unroll
            for (int j = 0; j < kAChunks; ++j) {
                const uint32_t off = static_cast<uint32_t>((tt + kSplitThreads * j) * 16);
                float4 hi, lo;
                split_tf32(av[j].x, hi.x, lo.x);
                split_tf32(av[j].y, hi.y, lo.y);
                split_tf32(av[j].z, hi.z, lo.z);
                split_tf32(av[j].w, hi.w, lo.w);
                sts128(a_big + off, hi);
                sts128(a_small + off, lo);
            }
            // B: the slice arrives as BK rows (k) of BN floats (n).  Column
            // n = bn becomes row bn of the K-major tiles: the 16-byte chunk of
            // k = 4c..4c+3 goes to chunk position c XOR the row's swizzle key,
            // address bits 7 and up of the row (bn mod 8 for 128-byte rows,
            // (bn / 2) mod 4 for 64-byte rows).
            // (PB: B's parts are already there, from the TMA.)
            if constexpr (!PB) {
#pragma unroll
                for (int c = 0; c < kBGroups; ++c) {
                    float4 hi, lo;
                    split_tf32(bv[c][0], hi.x, lo.x);
                    split_tf32(bv[c][1], hi.y, lo.y);
                    split_tf32(bv[c][2], hi.z, lo.z);
                    split_tf32(bv[c][3], hi.w, lo.w);
                    const int key = (bn * T::kRowBytes) >> 7;
                    const uint32_t off =
                        static_cast<uint32_t>(bn * T::kRowBytes + ((((bc0 + c) ^ key) & (BK / 4 - 1)) << 4));
                    sts128(b_big + off, hi);
                    sts128(b_small + off, lo);
                }
            }
            fence_proxy_async_smem();  // make the tiles visible to the tensor core
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(raw_empty(r));
                mbar_arrive(split_full(s));
            }
        }

        // Epilogue: accumulator row (32 * (warp % 4) + lane) lives in that
        // tensor-memory lane; the split warps sharing a lane quarter take
        // different 32-column chunks.
        // (timed_out is warp-uniform here: every wait above voted across the warp)
        if (!timed_out && nkt > 0 && mbar_wait_bounded_warp(acc_full, 0, tmo)) {
            tc_fence_after_sync();
            const int q = warp & 3;
            const int half = (warp - 2) / 4;  // which of the warps on this quarter
            constexpr int kChunksPerWarp = (BN / 32) / (kTcSplitWarps / 4);
            const int row = m0 + 32 * q + lane;
            float* crow = p.C + static_cast<long long>(row) * p.ldc;
            // (a later part of a split tile: its whole partial tile, rows and
            // columns beyond M and N included, into its workspace tile)
            float* wrow =
                second ? p.ws + ((static_cast<long long>(local) * (ks - 1) + part - 1) * T::kBM + 32 * q + lane) * BN
                       : nullptr;
            // C without 16-byte addressable rows: each 32 x 32 chunk passes
            // through a patch of the (now idle) split stages, 33 floats a row,
            // and goes out a row at a time, lane = column, so that a store
            // instruction writes 128 consecutive bytes instead of one float
            // in each of 32 rows.  (The MMAs that read the split stages have
            // completed: acc_full.)
            float* const patch =
                reinterpret_cast<float*>(smem_raw + (split(0) - raw_base)) + (warp - 2) * (32 * 33);
#pragma unroll
            for (int cc = 0; cc < kChunksPerWarp; ++cc) {
                const int ch = half * kChunksPerWarp + cc;
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(32 * ch), v);
                tmem_wait_ld();
                const int col = n0 + 32 * ch;
                if (second) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(wrow + 32 * ch + e) =
                            make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                        __uint_as_float(v[e + 3]));
                } else if (p.vec_store && col + 31 < p.N) {  // (warp-uniform)
                    if (row < p.M) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(crow + col + e) =
                                make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                            __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) patch[lane * 33 + e] = __uint_as_float(v[e]);
                    __syncwarp();
                    const int r0 = m0 + 32 * q;
                    for (int rr = 0; rr < 32 && r0 + rr < p.M; ++rr)
                        if (col + lane < p.N)
                            p.C[static_cast<long long>(r0 + rr) * p.ldc + col + lane] = patch[rr * 33 + lane];
                    __syncwarp();  // the patch is read before the next chunk overwrites it
                }
            }
        } else if (nkt > 0) {
            timed_out = true;
        }
    }

    if (timed_out) atomicOr(p.status, kTcStatusTimeout);
    if (ksplit) __threadfence();  // this thread's partial-tile stores, before the arrival below
    tc_fence_before_sync();
    const int any_timed_out = __syncthreads_or(timed_out ? 1 : 0);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, T::kTmemCols);
    }
    // K split: every part that stored its partial tile arrives on the tile's
    // counter; the CTA whose arrival is the last adds the parts into C.  No
    // CTA waits on another, and the sum does not depend on which CTA that is.
    if (ksplit && !any_timed_out) {
        if (threadIdx.x == 0) {
            const unsigned int prev = atomicAdd(p.split_count + local, 1u);
            *last_part = prev == static_cast<unsigned int>(ks - 1) ? 1 : 0;
            __threadfence();  // (the other parts' stores precede their arrivals)
        }
        __syncthreads();
        if (*last_part) tc_split_finish<BN>(p, local, ks, m0, n0);
    }
}

}  // namespace gb300
