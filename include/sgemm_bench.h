/*
 * sgemm_bench.h -- peak-rate microbenchmarks shipped with the library.
 *
 * They measure the two denominators of the roofline that bounds the matrix
 * multiply: the FP32 multiply-add rate of the CUDA cores and the HBM streaming
 * bandwidth.  They are measurement aids, not part of the product operation;
 * "Matrix multiplication performance optimisation", section 5 (performance
 * analysis), asks for every kernel to be judged against such ceilings.
 *
 * Both enqueue one kernel on `stream` (a cudaStream_t as void*) and return
 * without synchronising; the caller times them with CUDA events.  Return 0 on
 * success, 1 on invalid arguments, 3 if the launch failed.
 */
#ifndef GB300_SGEMM_BENCH_H
#define GB300_SGEMM_BENCH_H

#ifdef __cplusplus
extern "C" {
#endif

/* Independent FMA chains on every thread of `blocks` CTAs of 256 threads,
 * `iters` x 128 multiply-adds per thread (x2 when `paired`, which issues
 * fma.rn.f32x2).  `scratch` is a device buffer of blocks*256 floats that is
 * written only in a case that never happens (it keeps the chains live).
 * *flops_per_launch receives 2 x the multiply-adds the launch performs. */
int sgemm_bench_fma_peak(int paired, int blocks, int iters, float* scratch, void* stream,
                         double* flops_per_launch);

/* dst[0:n] = src[0:n] (device pointers, 16-byte aligned, n a multiple of 4),
 * grid-stride float4 copy over `blocks` CTAs of 256 threads.  Moves 8*n bytes. */
int sgemm_bench_copy(const float* src, float* dst, long long n, int blocks, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_SGEMM_BENCH_H */
