// Peak-rate microbenchmarks: the denominators of the roofline.
//
//  * FP32 FMA peak: every thread runs independent multiply-add chains, either
//    one FMA per instruction (FFMA) or two per instruction (fma.rn.f32x2);
//  * streaming copy: a grid-stride float4 copy, reporting read + write bytes.
//
// Exposed through include/sgemm_bench.h.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/sgemm_bench.h"

namespace gb300 {
namespace {

constexpr int kChains = 8;  // independent accumulators (pairs for the x2 form) per thread

__global__ void __launch_bounds__(256) peak_ffma_kernel(float* out, float a, float b, int iters) {
    float acc[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = static_cast<float>(threadIdx.x + c);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 16; ++u)
#pragma unroll
            for (int c = 0; c < kChains; ++c) acc[c] = fmaf(acc[c], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += acc[c];
    if (s == 1234.5f) out[blockIdx.x * blockDim.x + threadIdx.x] = s;  // keeps the chains live
}

__global__ void __launch_bounds__(256) peak_ffma2_kernel(float* out, float a, float b, int iters) {
    float2 acc[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = make_float2(threadIdx.x + c, threadIdx.x - c);
    const float2 aa = make_float2(a, a), bb = make_float2(b, b);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 16; ++u)
#pragma unroll
            for (int c = 0; c < kChains; ++c) acc[c] = __ffma2_rn(acc[c], aa, bb);
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += acc[c].x + acc[c].y;
    if (s == 1234.5f) out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void __launch_bounds__(256) copy_kernel(const float4* __restrict__ src, float4* __restrict__ dst,
                                                   long long n4) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
        dst[i] = src[i];
}

}  // namespace
}  // namespace gb300

extern "C" {

int sgemm_bench_fma_peak(int paired, int blocks, int iters, float* scratch, void* stream,
                         double* flops_per_launch) {
    if (blocks <= 0 || iters <= 0 || !scratch) return 1;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (paired)
        gb300::peak_ffma2_kernel<<<blocks, 256, 0, s>>>(scratch, 0.999f, 0.001f, iters);
    else
        gb300::peak_ffma_kernel<<<blocks, 256, 0, s>>>(scratch, 0.999f, 0.001f, iters);
    if (cudaGetLastError() != cudaSuccess) return 3;
    if (flops_per_launch)
        *flops_per_launch = 2.0 * static_cast<double>(blocks) * 256.0 * iters * 16.0 * gb300::kChains *
                            (paired ? 2.0 : 1.0);
    return 0;
}

int sgemm_bench_copy(const float* src, float* dst, long long n, int blocks, void* stream) {
    if (n < 0 || (n % 4) != 0 || blocks <= 0 || ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u))
        return 1;
    gb300::copy_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(src), reinterpret_cast<float4*>(dst), n / 4);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // extern "C"
