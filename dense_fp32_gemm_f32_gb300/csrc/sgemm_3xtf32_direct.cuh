// Three-product TF32 matrix multiply on the tensor cores, "direct-A" variant.
//
// Same arithmetic contract as the split-tile kernel in sgemm_3xtf32.cuh, with
// less shared-memory traffic per product:
//  * the big part of A is the FP32 tile exactly as the TMA lands it: the
//    tensor core reads the top 19 bits (sign, exponent, 10 mantissa bits) of
//    each 32-bit element, i.e. a_big = a with its low 13 bits cleared; the
//    split warps store only a_small = a - a_big (exact in FP32, at most 13
//    significant bits, of which the tensor core keeps 11: an error below
//    2^-20 |a|), element-wise in the same K-major swizzled layout;
//  * B still needs both parts stored: the tensor core reads TF32 operands
//    K-major (a layout with n innermost is not accepted for kind::tf32), so
//    B is transposed on the way, b_big = tf32(b), b_small = tf32(b - b_big);
//  * per k-step the three MMAs are A*B_small (A kept in the collector
//    buffer), A*B_big (A reused from the collector), A_small*B_big, so A is
//    read from shared memory once for two products.
// The dropped terms are below 2^-20 |a||b| per product, 20x inside the 5e-5
// contract; integer inputs in {-8..8} have zero small parts (exact).
//
// Pipeline (one CTA per 128 x 128 tile of C, 10 warps, 3 MMA stages of 64
// KiB and 2 raw-B slots of 16 KiB): warp 0 issues the TMA copy of the A slice
// into an MMA stage and of the B slice into a raw-B slot; warps 2..9 wait for
// both, write A_small, B_big and B_small into the stage, release the raw-B
// slot (`bfree`) and arrive on `ready`; warp 1 (lane 0) issues the 12 MMAs of
// the stage and commits them to `empty`, which frees the stage for the
// producer.  After the last stage the split warps read the accumulator from
// tensor memory and store C.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "sgemm_3xtf32_params.h"

namespace gb300 {

// The part of x below the TF32 precision the tensor core reads.
__device__ __forceinline__ float tf32_tail(float x) {
    return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

__global__ void __launch_bounds__(kTdThreads, 1)
    sgemm_3xtf32_direct_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                               const TcParams p) {
    constexpr int S = kTdStages;
    constexpr int RB = kTdRawBStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    // MMA stage layout: [raw A | A small | B big | B small], 16 KiB each;
    // then the raw-B slots.
    auto stage = [&](int st) { return base + static_cast<uint32_t>(st * kTdStageBytes); };
    auto raw_b_slot = [&](int rb) { return base + static_cast<uint32_t>(S * kTdStageBytes + rb * kTdTile); };
    const uint32_t bars = base + kTdRingBytes;
    auto full = [&](int st) { return bars + 8u * st; };                // raw A landed
    auto ready = [&](int st) { return bars + 8u * (S + st); };         // stored parts written
    auto empty = [&](int st) { return bars + 8u * (2 * S + st); };     // MMAs of the stage done
    auto bfull = [&](int rb) { return bars + 8u * (3 * S + rb); };     // raw B landed
    auto bfree = [&](int rb) { return bars + 8u * (3 * S + RB + rb); };  // raw B read
    const uint32_t acc_full = bars + 8u * (3 * S + 2 * RB);
    const uint32_t tmem_slot = acc_full + 8u;
    static_assert(8 * (3 * S + 2 * RB + 1) + 4 <= 256, "barrier area");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tile = static_cast<int>(blockIdx.x);
    const int n0 = (tile % p.tiles_n) * kTdBN;
    const int m0 = (tile / p.tiles_n) * kTdBM;
    const int nkt = p.num_k_tiles;
    const unsigned long long tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(full(st), 1);
            mbar_init(ready(st), kTdSplitWarps);
            mbar_init(empty(st), 1);
        }
        for (int rb = 0; rb < RB; ++rb) {
            mbar_init(bfull(rb), 1);
            mbar_init(bfree(rb), kTdSplitWarps);
        }
        mbar_init(acc_full, 1);
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTdTmemCols);
        tmem_relinquish_alloc_permit();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
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
            int issued_round[S], issued_round_b[RB];
#pragma unroll
            for (int st = 0; st < S; ++st) issued_round[st] = -1;
#pragma unroll
            for (int rb = 0; rb < RB; ++rb) issued_round_b[rb] = -1;
            const bool skip_here = p.skip_stage > 0 && tile == 0;
            for (int kt = 0; kt < nkt; ++kt) {
                const int st = kt % S, rb = kt % RB;
                const int round = kt / S, round_b = kt / RB;
                if ((round > 0 && !mbar_wait_bounded(empty(st), (round - 1) & 1, tmo)) ||
                    (round_b > 0 && !mbar_wait_bounded(bfree(rb), (round_b - 1) & 1, tmo))) {
                    timed_out = true;
                    break;
                }
                if (skip_here && kt == p.skip_stage - 1) continue;
                mbar_arrive_expect_tx(full(st), kTdTile);
                tma_load_2d(stage(st), &tmA, full(st), kt * kTdBK, m0);
                mbar_arrive_expect_tx(bfull(rb), kTdTile);
                tma_load_2d(raw_b_slot(rb), &tmB, bfull(rb), n0, kt * kTdBK);
                issued_round[st] = round;
                issued_round_b[rb] = round_b;
            }
            // drain: every issued copy has landed
            for (int st = 0; st < S; ++st)
                if (issued_round[st] >= 0 && !mbar_wait_bounded(full(st), issued_round[st] & 1, tmo))
                    timed_out = true;
            for (int rb = 0; rb < RB; ++rb)
                if (issued_round_b[rb] >= 0 && !mbar_wait_bounded(bfull(rb), issued_round_b[rb] & 1, tmo))
                    timed_out = true;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (int kt = 0; kt < nkt; ++kt) {
                const int st = kt % S;
                if (!mbar_wait_bounded(ready(st), (kt / S) & 1, tmo)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_big = stage(st), a_small = a_big + kTdTile;
                const uint32_t b_big = a_big + 2 * kTdTile, b_small = a_big + 3 * kTdTile;
#pragma unroll
                for (int kk = 0; kk < kTdBK / 8; ++kk) {  // k-steps of 8 TF32 = 32 bytes of each row
                    const uint32_t off = static_cast<uint32_t>(kk * 32);
                    const uint64_t da = umma_desc_kmajor_sw128(a_big + off);
                    const uint64_t db = umma_desc_kmajor_sw128(b_big + off);
                    umma_tf32_keep_a(tmem, da, umma_desc_kmajor_sw128(b_small + off), kTcIdesc, kt > 0 || kk > 0);
                    umma_tf32_reuse_a(tmem, da, db, kTcIdesc, true);
                    umma_tf32(tmem, umma_desc_kmajor_sw128(a_small + off), db, kTcIdesc, true);
                }
                umma_commit(empty(st));  // the stage is free once these MMAs are done
            }
            umma_commit(acc_full);  // arrives when every MMA above has completed
            if (!mbar_wait_bounded(acc_full, 0, tmo)) timed_out = true;
        }
    } else {
        // ------------------------------------------------------------ split + epilogue
        const int tt = threadIdx.x - 64;
        constexpr int kSplitThreads = 32 * kTdSplitWarps;
        constexpr int kAChunks = kTdTile / 16 / kSplitThreads;          // 16-byte A chunks per thread
        constexpr int kBGroups = (kTdBN * kTdBK / 4) / kSplitThreads;   // (column, 4-k) groups per thread
        const int bn = tt % kTdBN;
        const int bc0 = (tt / kTdBN) * kBGroups;
        for (int kt = 0; kt < nkt; ++kt) {
            const int st = kt % S, rb = kt % RB;
            if (!mbar_wait_bounded_warp(full(st), (kt / S) & 1, tmo) ||
                !mbar_wait_bounded_warp(bfull(rb), (kt / RB) & 1, tmo)) {
                timed_out = true;
                break;
            }
            const uint32_t raw_a = stage(st), raw_b = raw_b_slot(rb);
            const uint32_t a_small = raw_a + kTdTile, b_big = raw_a + 2 * kTdTile, b_small = raw_a + 3 * kTdTile;
            // Loads first (their latencies overlap), then conversions and stores.
            float4 av[kAChunks];
#pragma unroll
            for (int j = 0; j < kAChunks; ++j) av[j] = lds128(raw_a + static_cast<uint32_t>((tt + kSplitThreads * j) * 16));
            float bv[kBGroups][4];
            const uint32_t bcol = raw_b + static_cast<uint32_t>(bn * 4);
#pragma unroll
            for (int c = 0; c < kBGroups; ++c)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    asm volatile("ld.shared.f32 %0, [%1];"
                                 : "=f"(bv[c][i])
                                 : "r"(bcol + static_cast<uint32_t>((4 * (bc0 + c) + i) * kTdBN * 4)));
            // A: small parts, element-wise in the TMA's K-major swizzled layout.
#pragma unroll
            for (int j = 0; j < kAChunks; ++j)
                sts128(a_small + static_cast<uint32_t>((tt + kSplitThreads * j) * 16),
                       make_float4(tf32_tail(av[j].x), tf32_tail(av[j].y), tf32_tail(av[j].z), tf32_tail(av[j].w)));
            // B: column bn becomes row bn of the K-major tiles; the 16-byte
            // chunk of k = 4c..4c+3 goes to chunk position c ^ (bn mod 8).
#pragma unroll
            for (int c = 0; c < kBGroups; ++c) {
                float4 hi, lo;
                hi.x = to_tf32_rna(bv[c][0]);
                hi.y = to_tf32_rna(bv[c][1]);
                hi.z = to_tf32_rna(bv[c][2]);
                hi.w = to_tf32_rna(bv[c][3]);
                lo.x = to_tf32_rna(bv[c][0] - hi.x);
                lo.y = to_tf32_rna(bv[c][1] - hi.y);
                lo.z = to_tf32_rna(bv[c][2] - hi.z);
                lo.w = to_tf32_rna(bv[c][3] - hi.w);
                const uint32_t off = static_cast<uint32_t>(bn * 128 + ((((bc0 + c) ^ bn) & 7) << 4));
                sts128(b_big + off, hi);
                sts128(b_small + off, lo);
            }
            fence_proxy_async_smem();  // make the tiles visible to the tensor core
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bfree(rb));  // the raw B slot has been read (and used)
                mbar_arrive(ready(st));
            }
        }

        // Epilogue: accumulator row (32 * (warp % 4) + lane) is that tensor-
        // memory lane; the two split warps on a lane quarter take halves of
        // the columns.  (timed_out is warp-uniform: every wait above voted.)
        if (!timed_out && nkt > 0 && mbar_wait_bounded_warp(acc_full, 0, tmo)) {
            tc_fence_after_sync();
            const int q = warp & 3;
            const int half = (warp - 2) / 4;
            constexpr int kChunksPerWarp = (kTdBN / 32) / (kTdSplitWarps / 4);
            const int row = m0 + 32 * q + lane;
            float* crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll
            for (int cc = 0; cc < kChunksPerWarp; ++cc) {
                const int ch = half * kChunksPerWarp + cc;
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(32 * ch), r);
                tmem_wait_ld();
                const int col = n0 + 32 * ch;
                if (row < p.M) {
                    if (p.vec_store && col + 31 < p.N) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(crow + col + e) =
                                make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                            __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (col + e < p.N) crow[col + e] = __uint_as_float(r[e]);
                    }
                }
            }
        } else if (nkt > 0) {
            timed_out = true;
        }
    }

    if (timed_out) atomicOr(p.status, kTcStatusTimeout);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTdTmemCols);
    }
}

}  // namespace gb300
