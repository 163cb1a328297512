// Host-side registry of the compiled kernel variants (internal to the library).
#pragma once

#include <cuda_runtime.h>

namespace gb300 {

struct KernelEntry {
    const void* fn;   // host stub of the __global__ function, or nullptr if not built
    int smem_bytes;   // dynamic shared memory the launch needs
    int threads;      // threads per CTA
    bool tma_store = false;  // FFMA kernels: can write C by tensor-map stores (FfmaParams::tma_store)
};

// FFMA kernels fed by tensor-map bulk copies; stages in {1,2,3,4,5,6}, math 1 = FFMA, 2 = paired FFMA.
KernelEntry ffma_kernel_tma(int stages, int math);
// The same with the producer in a warpgroup of its own and the register split
// (producer 40, consumers 232 registers per thread); launched only when the
// kernel was built with exactly 168 registers per thread.
KernelEntry ffma_kernel_tma_wg(int stages, int math);
// 128 x 256 tiles (8 x 16 accumulators per thread) with the producer
// warpgroup and the register split; stages in {2,3,4}.
KernelEntry ffma_kernel_tma_wide(int stages, int math);
// The same on A stored transposed (K x M): 2 stages, paired FMA.
KernelEntry ffma_kernel_tma_wide_amn(int stages, int math);
// FFMA kernels with A transposed in shared memory by a second producer warp
// (128 x 128 tiles, stages in {2,3,4}; scaled epilogue: 2 stages, paired FMA);
// `edge`: the instantiations that compute a thin column edge (FfmaParams ec;
// paired FMA, plain epilogue).
KernelEntry ffma_kernel_tma_x(int stages, int math, bool scaled, bool edge = false);
// Fused-producer FFMA kernels: 4-warp CTAs (no producer warp; thread 0
// issues the TMA copies), 128 x 64 tiles, two CTAs per SM; stages in {2,3,4}.
KernelEntry ffma_kernel_tma_fused(int stages, int math);
// The scaled-epilogue FFMA kernels of the general entry: (TMA, 2 stages) and
// (cp.async, 4 stages), paired FMA, 128 x 128 tiles; nullptr otherwise.
KernelEntry ffma_kernel_scaled(int producer, int stages, int math);
// Transposed-A FFMA kernels (A stored K x M): TMA producer, 2 stages, paired
// FMA, 128 x 128 tiles; `scaled` selects the scaled epilogue.
KernelEntry ffma_kernel_amn(int stages, int math, bool scaled);
// FFMA kernels with A transposed in shared memory on 16-deep K slices
// (128 x 128 tiles, paired FMA, plain epilogue); stages in {2,3,4,6}.
KernelEntry ffma_kernel_tma_x16(int stages, int math);
// FFMA kernels on B stored N x K (op(B) = B^T, read in place and transposed
// in shared memory by a producer warp): A stored M x K (transposed in shared
// memory too) or, with `a_mn`, K x M; 2 stages, paired FMA, 128 x 128 tiles;
// `scaled` selects the scaled epilogue.
KernelEntry ffma_kernel_bnk(bool a_mn, bool scaled);
// FFMA kernels on residue-class tensor maps (operands of any alignment, read
// in place: four maps per operand, one per class of rows mod 4, and a
// B-shifting producer warp); 128 x 128 tiles, paired FMA; plain epilogue on
// stages {2,3,4}, `scaled` (the general entry's epilogue) on 2; `edge` as for
// ffma_kernel_tma_x.
KernelEntry ffma_kernel_res(int stages, int math, bool scaled = false, bool edge = false);
// FFMA kernels fed by loader warps (operands of any alignment, no tensor
// maps): 128 x 128 tiles, paired FMA, plain epilogue; stages {2,3,4}.
KernelEntry ffma_kernel_ldg(int stages, int math);
// FFMA kernels fed by 4-byte cp.async (any alignment); stages in {2,4}.
KernelEntry ffma_kernel_cpasync(int stages, int math);
// Three-product TF32 kernel on the tensor cores (TMA-fed, 128 x 128 tiles,
// all four TF32 parts stored in shared memory).
KernelEntry tf32x3_kernel();
// Direct-A three-product TF32 kernel: A's big part read from the TMA tile,
// only A's small part and B's two parts stored (128 x 128 tiles).
KernelEntry tf32x3_direct_kernel();
// The split-tile kernel on 128 x 256 tiles with K-slices of 16 (64-byte
// swizzled operand rows, 256 tensor-memory columns).
KernelEntry tf32x3_wide_kernel();
// The split-tile kernel (128 x 128 tiles) on residue-class tensor maps:
// operands of any alignment read in place; 2 raw stages.
KernelEntry tf32x3_res_kernel();

// Copies up to two operands (a null dst skips one): `rows` rows of `cols`
// floats from `src` (pitch ld_src floats, any alignment) to `dst` (pitch
// ld_dst floats: a multiple of 4, >= cols; 16-byte aligned base), zero-filling
// each row's padding; one launch, enqueued on `stream`.
int pack_rows(const float* src0, long long ld_src0, float* dst0, long long ld_dst0, int rows0, int cols0,
              const float* src1, long long ld_src1, float* dst1, long long ld_dst1, int rows1, int cols1,
              cudaStream_t stream);
// Transposing copies (a null dst skips one): dst (rows x cols, pitch ld_dst:
// a multiple of 4, >= cols; 16-byte aligned base) = the transpose of src
// (cols x rows, pitch ld_src >= rows), zero-filling each row's padding; one
// launch, enqueued on `stream`.
int transpose_rows(const float* src0, long long ld_src0, float* dst0, long long ld_dst0, int rows0, int cols0,
                   const float* src1, long long ld_src1, float* dst1, long long ld_dst1, int rows1, int cols1,
                   cudaStream_t stream);
// Small-problem FFMA kernel: one 8-warp CTA per 32 x 32 tile of C (grid
// ceil(N / 32) x ceil(M / 32)), K split across the warps in 32-deep chunks
// and the partials summed in a fixed order; bounds-checked 4-byte loads (any
// alignment).  `a_mn`: A stored transposed (K x M); `scaled`: C = alpha A B +
// beta C (beta == 0: C not read).
constexpr int kSmallTile = 32;
constexpr int kSmallWarps = 8;
constexpr int kSmallSmemBytes = kSmallWarps * (kSmallTile * (kSmallTile + 4) + kSmallTile * kSmallTile) * 4;
struct SmallParams {
    int M, N, K;
    const float* A;
    long long lda;
    const float* B;
    long long ldb;
    float* C;
    long long ldc;
    float alpha, beta;
};
KernelEntry small_kernel(bool a_mn, bool scaled);
// B's TF32 parts, transposed: big (N x K, pitch ld_out: a multiple of 4, >= K;
// 16-byte aligned base) = tf32(B^T), small = tf32(B^T - big); zeros in the
// padding columns; B (K x N, pitch ldb) of any alignment.  One launch on `stream`.
int split_transpose_b(const float* B, long long ldb, int K, int N, float* big, float* small, long long ld_out,
                      cudaStream_t stream);
// The split-tile kernel on 128 x 256 tiles with B's TF32 parts pre-split by
// split_transpose_b (loaded by the TMA; the kernel splits A only).
KernelEntry tf32x3_wide_pb_kernel();
// C = beta * C over M x N with pitch ldc (beta == 0: zeros, C not read).
int scale_c(float* C, long long ldc, int M, int N, float beta, cudaStream_t stream);

}  // namespace gb300
