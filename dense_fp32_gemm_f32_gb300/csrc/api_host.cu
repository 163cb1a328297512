// The host-buffer entry sgemm_f32_host: copies in and out on the library's
// copy streams, overlapped with the products of row blocks and K chunks.
#include "api_internal.h"

namespace gb300 {
namespace detail {

// Rows [r0, r0 + rows) of a rows x cols float matrix, pitch ld_src -> pitch
// ld_dst, as one (2-D when pitched) asynchronous copy.
cudaError_t copy_rows(float* dst, long long ld_dst, const float* src, long long ld_src, long long rows,
                      long long cols, cudaMemcpyKind kind, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (ld_dst == cols && ld_src == cols)
        return cudaMemcpyAsync(dst, src, static_cast<size_t>(rows * cols) * 4, kind, s);
    return cudaMemcpy2DAsync(dst, static_cast<size_t>(ld_dst) * 4, src, static_cast<size_t>(ld_src) * 4,
                             static_cast<size_t>(cols) * 4, static_cast<size_t>(rows), kind, s);
}

// Host-buffer form (see sgemm_f32_host): pitched device copies of A, B, C
// from the pool (rows of ceil(width / 4) x 4 floats, so that the tensor maps
// can always read them).  A and C move in row blocks so that block i's
// product overlaps block i+1's copy in and block i-1's copy out; B moves in K
// chunks, and the first block's product is split the same way (accumulating
// into C), so that the first product starts after A's first block and B's
// first chunk rather than after all of B.
int run_host(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
             void* stream) {
    int rc = validate(M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    int dev = 0;
    DeviceState* st = nullptr;
    rc = current_device(&dev, &st);
    if (rc != SGEMM_OK) return rc;
    // The copy streams and the events of the pipeline, made once per device.
    // Calls share them, so one call enqueues at a time (host_mu); reusing the
    // events is safe because a stream's wait on an event waits for the event's
    // last record at the time the wait is enqueued.
    std::call_once(st->copy_once, [&] {
        bool made = cudaStreamCreateWithFlags(&st->copy_in, cudaStreamNonBlocking) == cudaSuccess &&
                    cudaStreamCreateWithFlags(&st->copy_out, cudaStreamNonBlocking) == cudaSuccess;
        for (int e = 0; e < kHostEvents && made; ++e)
            made = cudaEventCreateWithFlags(&st->host_ev[e], cudaEventDisableTiming) == cudaSuccess;
        if (!made) {
            (void)cudaGetLastError();
            st->copy_in = st->copy_out = nullptr;
        }
    });
    if (!st->copy_in || !st->copy_out) return SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(st->host_mu);
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaMemPool_t pool = workspace_pool(dev, *st);
    if (!pool) return SGEMM_ERR_CUDA;

    // Row blocks: whole 128-row tiles, up to 8 blocks of >= 512 rows; one
    // block below 2^32 flop (the copies then run before and after the
    // product).  K chunks of B (multiples of 32): 4 when blocked and K >= 1024.
    constexpr int kMaxBlk = kHostMaxBlk, kMaxKc = kHostMaxKc;
    const bool big = 2.0 * static_cast<double>(M) * N * K >= 4294967296.0;
    const int nblk = big ? static_cast<int>(std::min<long long>(kMaxBlk, (static_cast<long long>(M) + 511) / 512)) : 1;
    const long long rows_blk = ((static_cast<long long>(M) + nblk - 1) / nblk + kBM - 1) / kBM * kBM;
    const int nkc = (big && nblk > 1 && K >= 1024) ? kMaxKc : 1;
    auto k_at = [&](int c) -> long long {
        return c >= nkc ? K : (static_cast<long long>(K) * c / nkc) / 32 * 32;
    };

    const long long K4 = (static_cast<long long>(K) + 3) / 4 * 4;
    const long long N4 = (static_cast<long long>(N) + 3) / 4 * 4;
    if (K4 > 0x7fffffffLL || N4 > 0x7fffffffLL) return SGEMM_ERR_INVALID_ARG;
    const size_t bytes_a = (static_cast<size_t>(M) * K4 * 4 + 255) & ~size_t{255};
    const size_t bytes_b = (static_cast<size_t>(K) * N4 * 4 + 255) & ~size_t{255};
    const size_t bytes_c = static_cast<size_t>(M) * N4 * 4;
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, bytes_a + bytes_b + bytes_c, pool, cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    float* dA = static_cast<float*>(ws);
    float* dB = reinterpret_cast<float*>(static_cast<char*>(ws) + bytes_a);
    float* dC = reinterpret_cast<float*>(static_cast<char*>(ws) + bytes_a + bytes_b);
    const int lda_d = static_cast<int>(K4), ldb_d = static_cast<int>(N4), ldc_d = static_cast<int>(N4);

    cudaEvent_t* const ev = st->host_ev;
    const cudaEvent_t ev_start = ev[0], ev_in_end = ev[1], ev_out_end = ev[2];
    cudaEvent_t* const ev_a = ev + 3;                 // [kMaxBlk]
    cudaEvent_t* const ev_done = ev + 3 + kMaxBlk;    // [kMaxBlk]
    cudaEvent_t* const ev_b = ev + 3 + 2 * kMaxBlk;   // [kMaxKc]
    // The copy streams start after the workspace exists (stream order of cs).
    bool ok = cudaEventRecord(ev_start, cs) == cudaSuccess &&
         cudaStreamWaitEvent(st->copy_in, ev_start, 0) == cudaSuccess &&
         cudaStreamWaitEvent(st->copy_out, ev_start, 0) == cudaSuccess;

    // Copies in, in the order the products need them: A's first block, B's
    // chunks, A's other blocks.
    auto copy_a = [&](int i) {
        const long long r0 = i * rows_blk, rows = std::min<long long>(rows_blk, M - r0);
        return rows <= 0 || (copy_rows(dA + r0 * K4, K4, A + r0 * lda, lda, rows, K, cudaMemcpyHostToDevice,
                                       st->copy_in) == cudaSuccess &&
                             cudaEventRecord(ev_a[i], st->copy_in) == cudaSuccess);
    };
    ok = ok && copy_a(0);
    for (int c = 0; c < nkc && ok; ++c)
        ok = copy_rows(dB + k_at(c) * N4, N4, B + k_at(c) * ldb, ldb, k_at(c + 1) - k_at(c), N,
                       cudaMemcpyHostToDevice, st->copy_in) == cudaSuccess &&
             cudaEventRecord(ev_b[c], st->copy_in) == cudaSuccess;
    for (int i = 1; i < nblk && ok; ++i) ok = copy_a(i);

    // Products on cs, copies out on copy_out.
    Scale accumulate;  // C += A_chunk B_chunk for the first block's later K chunks
    accumulate.alpha = 1.f;
    accumulate.beta = 1.f;
    for (int i = 0; i < nblk && ok && rc == SGEMM_OK; ++i) {
        const long long r0 = i * rows_blk, rows = std::min<long long>(rows_blk, M - r0);
        if (rows <= 0) break;
        ok = cudaStreamWaitEvent(cs, ev_a[i], 0) == cudaSuccess;
        const int chunks = i == 0 ? nkc : 1;
        for (int c = 0; c < chunks && ok && rc == SGEMM_OK; ++c) {
            const long long k0 = i == 0 ? k_at(c) : 0, k1 = i == 0 ? k_at(c + 1) : K;
            ok = cudaStreamWaitEvent(cs, ev_b[i == 0 ? c : nkc - 1], 0) == cudaSuccess;
            if (ok)
                rc = run_ffma(static_cast<int>(rows), N, static_cast<int>(k1 - k0), dA + r0 * K4 + k0, lda_d,
                              dB + k0 * N4, ldb_d, dC + r0 * N4, ldc_d, stream, nullptr, c > 0 ? &accumulate : nullptr);
        }
        if (!ok || rc != SGEMM_OK) break;
        ok = cudaEventRecord(ev_done[i], cs) == cudaSuccess &&
             cudaStreamWaitEvent(st->copy_out, ev_done[i], 0) == cudaSuccess &&
             copy_rows(C + r0 * ldc, ldc, dC + r0 * N4, N4, rows, N, cudaMemcpyDeviceToHost, st->copy_out) ==
                 cudaSuccess;
    }
    // cs resumes (and the workspace returns to the pool) after every copy in
    // and out, also after a failure, so that nothing in flight uses freed
    // memory.
    const bool joined = cudaEventRecord(ev_in_end, st->copy_in) == cudaSuccess &&
                        cudaEventRecord(ev_out_end, st->copy_out) == cudaSuccess &&
                        cudaStreamWaitEvent(cs, ev_in_end, 0) == cudaSuccess &&
                        cudaStreamWaitEvent(cs, ev_out_end, 0) == cudaSuccess;
    if (!ok || !joined) (void)cudaGetLastError();
    if (!joined) {
        (void)cudaStreamSynchronize(st->copy_in);
        (void)cudaStreamSynchronize(st->copy_out);
    }
    (void)cudaFreeAsync(ws, cs);
    if (rc != SGEMM_OK) return rc;
    return ok ? SGEMM_OK : SGEMM_ERR_CUDA;
}

}  // namespace detail
}  // namespace gb300
