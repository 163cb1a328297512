// Small-problem FFMA kernel: C = alpha * A B (+ beta * C) for products too
// small to fill the GPU with 128 x 128 tiles (256^3 has four such tiles, and
// one SM needs about 2 us for each 128 x 128 x 32 slice of one).  There the
// first load's latency and the per-SM work, not the FP32 pipe, set the time,
// so this kernel spreads the product over many small CTAs and keeps each
// CTA's critical path short:
//  * one CTA of 8 warps per 32 x 32 tile of C; warp w takes the K-chunks
//    w, w + 8, w + 16, ... of 32 and accumulates its own 32 x 32 partial,
//    a 4 x 8 block per lane (rows tm + 8i, columns 8 tn .. 8 tn + 7);
//  * operands are read with bounds-checked 4-byte loads (any alignment or
//    leading dimension; zeros past M, N and K), coalesced along the stored
//    rows, into registers one chunk ahead of the multiply-adds;
//  * each chunk passes through the warp's own shared-memory buffers (A as
//    [m][k] with a 36-float pitch, so that the 16-byte reads of 4 k values
//    of rows tm + 8i hit 8 different bank groups; B as [k][n]);
//  * the 8 partials are summed in warp order through shared memory, so the
//    result does not depend on timing.
// The pages' register-tiled kernels (a thread computing a block of C from
// shared-memory tiles) in a shape chosen for latency rather than throughput.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace gb300 {
namespace {

constexpr int kSmT = kSmallTile;                        // BM = BN = BK
constexpr int kSmAPitch = kSmT + 4;                     // floats per A row (m) in shared memory
constexpr int kSmWarpFloats = kSmT * kSmAPitch + kSmT * kSmT;  // A [m][k] + B [k][n]
constexpr int kSmThreads = 32 * kSmallWarps;
static_assert(kSmT == 32, "one lane per row element of a chunk");
static_assert(kSmT * kSmT <= kSmWarpFloats, "a warp's partial tile fits in its buffers");
static_assert((kSmWarpFloats * 4) % 16 == 0, "16-byte aligned warp buffers");
static_assert(kSmT * kSmT == 4 * kSmThreads, "four outputs of the reduction per thread");

// AT: A stored transposed (K x M, element (m, k) at A[k * lda + m]).
template <bool AT, bool SCALED>
__global__ void __launch_bounds__(kSmThreads) sgemm_small_kernel(const SmallParams p) {
    extern __shared__ float4 smem4[];
    float* const smem = reinterpret_cast<float*>(smem4);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float* const As = smem + warp * kSmWarpFloats;  // [m][k], pitch kSmAPitch
    float* const Bs = As + kSmT * kSmAPitch;        // [k][n], pitch kSmT
    const int m0 = static_cast<int>(blockIdx.y) * kSmT;
    const int n0 = static_cast<int>(blockIdx.x) * kSmT;
    const int nch = (p.K + kSmT - 1) / kSmT;
    const int tm = lane >> 2;  // rows tm + 8 i
    const int tn = lane & 3;   // columns 8 tn + j

    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    // Chunk c in registers: ra[r] = A(m0 + r, k0 + lane) (A as stored) or
    // A(m0 + lane, k0 + r) (A transposed); rb[r] = B(k0 + r, n0 + lane).
    float ra[kSmT], rb[kSmT];
    auto load = [&](int c) {
        const int k0 = c * kSmT;
#pragma unroll
        for (int r = 0; r < kSmT; ++r) {
            const int m = AT ? m0 + lane : m0 + r;
            const int k = AT ? k0 + r : k0 + lane;
            ra[r] = (m < p.M && k < p.K)
                        ? __ldg(AT ? p.A + static_cast<long long>(k) * p.lda + m : p.A + static_cast<long long>(m) * p.lda + k)
                        : 0.f;
        }
#pragma unroll
        for (int r = 0; r < kSmT; ++r) {
            const int k = k0 + r, n = n0 + lane;
            rb[r] = (k < p.K && n < p.N) ? __ldg(p.B + static_cast<long long>(k) * p.ldb + n) : 0.f;
        }
    };

    int c = warp;
    if (c < nch) load(c);
    for (; c < nch; c += kSmallWarps) {
        __syncwarp();  // the previous chunk's reads of the buffers are done
#pragma unroll
        for (int r = 0; r < kSmT; ++r) {
            if (AT)
                As[lane * kSmAPitch + r] = ra[r];
            else
                As[r * kSmAPitch + lane] = ra[r];
            Bs[r * kSmT + lane] = rb[r];
        }
        __syncwarp();
        if (c + kSmallWarps < nch) load(c + kSmallWarps);  // next chunk in flight during the multiply-adds
#pragma unroll
        for (int kk = 0; kk < kSmT; kk += 4) {
            float4 a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(As + (tm + 8 * i) * kSmAPitch + kk);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 b0 = *reinterpret_cast<const float4*>(Bs + (kk + q) * kSmT + 8 * tn);
                const float4 b1 = *reinterpret_cast<const float4*>(Bs + (kk + q) * kSmT + 8 * tn + 4);
                const float bq[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float aq = q == 0 ? a[i].x : q == 1 ? a[i].y : q == 2 ? a[i].z : a[i].w;
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(aq, bq[j], acc[i][j]);
                }
            }
        }
    }

    // The warp's partial, [m][n] with pitch kSmT, into its own buffers.
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float* row = As + (tm + 8 * i) * kSmT + 8 * tn;
        *reinterpret_cast<float4*>(row) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        *reinterpret_cast<float4*>(row + 4) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    __syncthreads();
    // Thread t finishes elements t, t + 256, ... of the tile (consecutive
    // threads, consecutive columns): the sum over warps 0..7 in order.
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int o = static_cast<int>(threadIdx.x) + kSmThreads * q;
        const int m = o / kSmT, n = o % kSmT;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kSmallWarps; ++w) s += smem[w * kSmWarpFloats + m * kSmT + n];
        const int gm = m0 + m, gn = n0 + n;
        if (gm < p.M && gn < p.N) {
            float* out = p.C + static_cast<long long>(gm) * p.ldc + gn;
            if (SCALED)
                *out = p.beta == 0.f ? p.alpha * s : fmaf(p.alpha, s, p.beta * *out);
            else
                *out = s;
        }
    }
}

template <bool AT, bool SCALED>
KernelEntry entry() {
    return {reinterpret_cast<const void*>(&sgemm_small_kernel<AT, SCALED>), kSmallSmemBytes, kSmThreads};
}

}  // namespace

static_assert(kSmallSmemBytes == kSmallWarps * kSmWarpFloats * 4, "shared memory of the small kernel");

KernelEntry small_kernel(bool a_mn, bool scaled) {
    if (a_mn) return scaled ? entry<true, true>() : entry<true, false>();
    return scaled ? entry<false, true>() : entry<false, false>();
}

}  // namespace gb300
