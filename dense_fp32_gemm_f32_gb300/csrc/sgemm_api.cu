// C ABI of the library (include/sgemm.h): the entry points, which check their
// arguments and hand the work to the translation units declared in
// api_internal.h.
#include "api_internal.h"

using namespace gb300;
using namespace gb300::detail;

extern "C" {

int sgemm_f32(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
              void* stream) {
    return run_ffma(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr);
}

int sgemm_f32_ex(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                 void* stream, const sgemm_options* opt) {
    return run_ffma(M, N, K, A, lda, B, ldb, C, ldc, stream, opt);
}

int sgemm_f32_noalloc(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                      void* stream) {
    return run_ffma_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream);
}

int sgemm_f32_host(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                   void* stream) {
    return run_host(M, N, K, A, lda, B, ldb, C, ldc, stream);
}

int sgemm_f32_gemm(int transa, int transb, int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                   int ldb, float beta, float* C, int ldc, void* stream) {
    return run_gemm(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

int sgemm_3xtf32(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                 void* stream) {
    return run_3xtf32(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr);
}

int sgemm_3xtf32_ex(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                    void* stream, const sgemm_options* opt) {
    return run_3xtf32(M, N, K, A, lda, B, ldb, C, ldc, stream, opt);
}

int sgemm_check_status(void* stream) {
    int dev = 0;
    DeviceState* st = nullptr;
    const int rc = current_device(&dev, &st);
    if (rc != SGEMM_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (cudaMemcpy(&word, st->status_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(st->status_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    return (word & kStatusTimeout) ? SGEMM_ERR_TIMEOUT : SGEMM_OK;
}

const char* sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_OK: return "ok";
        case SGEMM_ERR_INVALID_ARG: return "invalid argument";
        case SGEMM_ERR_UNSUPPORTED: return "unsupported device or variant";
        case SGEMM_ERR_CUDA: return "CUDA error";
        case SGEMM_ERR_TIMEOUT: return "kernel wait timed out";
        case SGEMM_ERR_NOT_IMPLEMENTED: return "not implemented";
        default: return "unknown status";
    }
}

const char* sgemm_describe(int M, int N, int K, const float* A, int lda, const float* B, int ldb, const float* C,
                           int ldc) {
    if (validate(M, N, K, A, lda, B, ldb, C, ldc) != SGEMM_OK) return "invalid";
    int dev = 0;
    DeviceState* st = nullptr;
    if (current_device(&dev, &st) != SGEMM_OK) return "unavailable";
    if (M == 0 || N == 0) return "noop";
    if (small_problem(*st, M, N, K)) return "small/t32/w8";
    Plan pl;
    if (make_plan(*st, M, N, K, A, lda, B, ldb, nullptr, &pl) != SGEMM_OK) return "invalid";
    return describe_plan(pl);
}

}  // extern "C"
