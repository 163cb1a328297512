// Row repacking for operands whose rows the tensor maps cannot address.
//
// A tensor map needs a 16-byte aligned base and a row pitch that is a multiple
// of 16 bytes.  An operand without them (a leading dimension that is not a
// multiple of 4 floats, or a base off a 16-byte boundary) is copied once into
// a buffer whose pitch is the row width rounded up to 4 floats; the product
// then runs on the tensor-map path.  The copy is plain element moves, so the
// product's result is unchanged.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kernels.h"
#include "../../include/sgemm.h"

namespace gb300 {
namespace {

constexpr int kPackThreads = 256;

struct PackJob {
    const float* src;
    long long ld_src;
    float* dst;
    long long ld_dst;
    int rows, cols;
};

// Job blockIdx.z, rows [kPackRows * blockIdx.x, + kPackRows): dst row r,
// floats [c4, c4 + 4) <- src row r, the same columns (zeros past `cols`, i.e.
// in the pitch padding), for every 4-float group c4 of the dst row, threads
// striding along the row.  Reads are coalesced scalar loads (the source rows
// have any alignment), writes 16-byte stores; the loads of the CTA's rows
// are all issued before the first store, so that a CTA waits one memory
// round trip per group of rows rather than one per row.
constexpr int kPackRows = 4;

__global__ void __launch_bounds__(kPackThreads) pack_rows_kernel(const PackJob j0, const PackJob j1) {
    const PackJob& j = blockIdx.z == 0 ? j0 : j1;
    const long long r0 = static_cast<long long>(blockIdx.x) * kPackRows;
    if (r0 >= j.rows) return;
    const long long groups = j.ld_dst / 4;
    for (long long q = threadIdx.x; q < groups; q += kPackThreads) {
        const long long c4 = 4 * q;
        float4 v[kPackRows];
#pragma unroll
        for (int i = 0; i < kPackRows; ++i) {
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r0 + i >= j.rows) continue;
            const float* s = j.src + (r0 + i) * j.ld_src;
            if (c4 + 0 < j.cols) v[i].x = s[c4 + 0];
            if (c4 + 1 < j.cols) v[i].y = s[c4 + 1];
            if (c4 + 2 < j.cols) v[i].z = s[c4 + 2];
            if (c4 + 3 < j.cols) v[i].w = s[c4 + 3];
        }
#pragma unroll
        for (int i = 0; i < kPackRows; ++i)
            if (r0 + i < j.rows) *reinterpret_cast<float4*>(j.dst + (r0 + i) * j.ld_dst + c4) = v[i];
    }
}

// Transposing copy, job blockIdx.z: dst[r][c] = src[c][r] for r < rows,
// c < cols (dst is rows x cols with pitch ld_dst; src is cols x rows with
// pitch ld_src); dst's padding columns [cols, ld_dst) are zero-filled.  A
// 32 x 32 tile passes through shared memory with one padding column, so that
// both the reads (along src rows) and the writes (along dst rows) are
// coalesced and the column-wise shared-memory reads hit 32 different banks.
constexpr int kTile = 32;
constexpr int kTileRows = 8;

__global__ void __launch_bounds__(kTile* kTileRows) transpose_kernel(const PackJob j0, const PackJob j1) {
    __shared__ float tile[kTile][kTile + 1];
    const PackJob& j = blockIdx.z == 0 ? j0 : j1;
    const long long c0 = static_cast<long long>(blockIdx.x) * kTile;  // dst columns = src rows
    if (c0 >= j.ld_dst) return;
    const long long row_tiles = (j.rows + kTile - 1) / kTile;
    for (long long ty = blockIdx.y; ty < row_tiles; ty += gridDim.y) {
        const long long r0 = ty * kTile;  // dst rows = src columns
        for (int y = threadIdx.y; y < kTile; y += kTileRows) {
            const long long sr = c0 + y, sc = r0 + threadIdx.x;
            tile[y][threadIdx.x] = (sr < j.cols && sc < j.rows) ? j.src[sr * j.ld_src + sc] : 0.f;
        }
        __syncthreads();
        for (int y = threadIdx.y; y < kTile; y += kTileRows) {
            const long long dr = r0 + y, dc = c0 + threadIdx.x;
            if (dr < j.rows && dc < j.ld_dst) j.dst[dr * j.ld_dst + dc] = tile[threadIdx.x][y];
        }
        __syncthreads();
    }
}

bool job_ok(const PackJob& j) {
    return j.ld_dst >= j.cols && j.ld_dst % 4 == 0 && (reinterpret_cast<uintptr_t>(j.dst) & 15u) == 0;
}

}  // namespace

int pack_rows(const float* src0, long long ld_src0, float* dst0, long long ld_dst0, int rows0, int cols0,
              const float* src1, long long ld_src1, float* dst1, long long ld_dst1, int rows1, int cols1,
              cudaStream_t stream) {
    PackJob j[2] = {{src0, ld_src0, dst0, ld_dst0, rows0, cols0}, {src1, ld_src1, dst1, ld_dst1, rows1, cols1}};
    int n = 0;
    PackJob use[2];
    for (const PackJob& x : j)
        if (x.dst && x.rows > 0 && x.cols > 0) {
            if (!job_ok(x)) return SGEMM_ERR_INVALID_ARG;
            use[n++] = x;
        }
    if (n == 0) return SGEMM_OK;
    if (n == 1) use[1] = use[0];
    long long gx = 0;
    for (int i = 0; i < n; ++i) {
        const long long x = (static_cast<long long>(use[i].rows) + kPackRows - 1) / kPackRows;
        gx = x > gx ? x : gx;
    }
    if (gx > 0x7fffffffLL) return SGEMM_ERR_INVALID_ARG;
    pack_rows_kernel<<<dim3(static_cast<unsigned>(gx), 1, static_cast<unsigned>(n)), kPackThreads, 0, stream>>>(
        use[0], use[1]);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}

int transpose_rows(const float* src0, long long ld_src0, float* dst0, long long ld_dst0, int rows0, int cols0,
                   const float* src1, long long ld_src1, float* dst1, long long ld_dst1, int rows1, int cols1,
                   cudaStream_t stream) {
    PackJob j[2] = {{src0, ld_src0, dst0, ld_dst0, rows0, cols0}, {src1, ld_src1, dst1, ld_dst1, rows1, cols1}};
    int n = 0;
    PackJob use[2];
    for (const PackJob& x : j)
        if (x.dst && x.rows > 0 && x.cols > 0) {
            if (!job_ok(x) || x.ld_src < x.rows) return SGEMM_ERR_INVALID_ARG;
            use[n++] = x;
        }
    if (n == 0) return SGEMM_OK;
    if (n == 1) use[1] = use[0];
    long long gx = 0, gy = 0;
    for (int i = 0; i < n; ++i) {
        gx = std::max(gx, (use[i].ld_dst + kTile - 1) / kTile);
        gy = std::max(gy, std::min<long long>((use[i].rows + kTile - 1) / kTile, 65535));
    }
    if (gx > 0x7fffffffLL) return SGEMM_ERR_INVALID_ARG;
    transpose_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(n)),
                       dim3(kTile, kTileRows), 0, stream>>>(use[0], use[1]);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}

namespace {

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// B (K x N, pitch ldb, any alignment) -> its TF32 parts transposed, N x K
// with pitch ld_out: big[n][k] = tf32(b), small[n][k] = tf32(b - big) (the
// same split as the tensor-core kernels' split warps), zeros in the padding
// columns k in [K, ld_out).  32 x 32 tiles through shared memory with one
// padding column (coalesced reads along n, writes along k); blocks walk the
// K direction in steps of gridDim.y.
__global__ void __launch_bounds__(kTile* kTileRows)
    split_transpose_kernel(const float* B, long long ldb, int K, int N, float* big, float* small, long long ld_out) {
    __shared__ float tile[kTile][kTile + 1];
    const int n0 = static_cast<int>(blockIdx.x) * kTile;
    for (long long k0 = static_cast<long long>(blockIdx.y) * kTile; k0 < ld_out;
         k0 += static_cast<long long>(gridDim.y) * kTile) {
#pragma unroll
        for (int j = 0; j < kTile / kTileRows; ++j) {
            const long long k = k0 + threadIdx.y + kTileRows * j;
            const int n = n0 + static_cast<int>(threadIdx.x);
            tile[threadIdx.y + kTileRows * j][threadIdx.x] = (k < K && n < N) ? B[k * ldb + n] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kTile / kTileRows; ++j) {
            const int n = n0 + static_cast<int>(threadIdx.y) + kTileRows * j;
            const long long k = k0 + threadIdx.x;
            if (n < N && k < ld_out) {
                const float v = tile[threadIdx.x][threadIdx.y + kTileRows * j];
                const float hi = tf32_rna(v);
                big[static_cast<long long>(n) * ld_out + k] = hi;
                small[static_cast<long long>(n) * ld_out + k] = tf32_rna(v - hi);
            }
        }
        __syncthreads();
    }
}

}  // namespace

int split_transpose_b(const float* B, long long ldb, int K, int N, float* big, float* small, long long ld_out,
                      cudaStream_t stream) {
    if (K <= 0 || N <= 0) return SGEMM_OK;
    if (ld_out < K || ld_out % 4 != 0 || ldb < N) return SGEMM_ERR_INVALID_ARG;
    const long long gx = (static_cast<long long>(N) + kTile - 1) / kTile;
    const long long gy = std::min<long long>((ld_out + kTile - 1) / kTile, 65535);
    if (gx > 0x7fffffffLL) return SGEMM_ERR_INVALID_ARG;
    split_transpose_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), dim3(kTile, kTileRows), 0,
                             stream>>>(B, ldb, K, N, big, small, ld_out);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}

namespace {

// C = beta * C over M x N (pitch ldc); beta == 0 writes zeros without reading.
__global__ void __launch_bounds__(256) scale_kernel(float* C, long long ldc, int M, int N, float beta) {
    const long long c = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
    if (c >= N) return;
    for (long long r = blockIdx.y; r < M; r += gridDim.y) {
        float* p = C + r * ldc + c;
        *p = beta == 0.f ? 0.f : beta * *p;
    }
}

}  // namespace

int scale_c(float* C, long long ldc, int M, int N, float beta, cudaStream_t stream) {
    if (M <= 0 || N <= 0) return SGEMM_OK;
    const long long gx = (static_cast<long long>(N) + 255) / 256;
    const int gy = M < 65535 ? M : 65535;
    scale_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), 256, 0, stream>>>(C, ldc, M, N, beta);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}

}  // namespace gb300
