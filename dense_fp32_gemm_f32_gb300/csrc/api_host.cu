// The host-buffer entry sgemm_f32_host: copies in and out on the library's
// copy streams, overlapped with the products of K chunks and row blocks.
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
// can always read them).
//
// Schedule of products of 2^32 flop and more.  The host link moves far fewer
// bytes per second than the product consumes (measured on GB300: ~210 GB/s
// in, ~195 GB/s out; a 4096 x 4096 output consumes a column of A and a row
// of B, 32 KB, every 0.5 us), so no product may wait for whole operands.  K
// is cut into chunks that grow (to 1/32, 5/32, 1/2 and all of K): chunk c's
// columns of A and rows of B cross the link together, and the product
// C (+)= A[:, c] B[c, :] over all rows starts once they are in, while the
// next chunk crosses.  The first chunk is short, so that the first product
// starts early; each later chunk is in before the product of the one before
// it ends (measured on GB300: pitched copies of 512-byte rows run at 131
// GB/s, of 6 KB rows and more at 203-208 GB/s).  The last chunk's product
// runs in row blocks that shrink towards the end (to 5/8, 13/16, 15/16 and
// all of the rows), each block's
// rows of C going back over the link while the next block computes, so that
// only the last, small block of C crosses after the last product.  Smaller
// products run as one block: copies in, product, copy out.
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

    // K chunks (boundaries multiples of 32) and the row blocks of the last
    // chunk (boundaries multiples of 128 rows); empty ones are dropped.
    const bool big = 2.0 * static_cast<double>(M) * N * K >= 4294967296.0;
    long long kb[kHostMaxKc + 1] = {0};
    int nkc = 0;
    {
        const int den = 32, num[kHostMaxKc] = {1, 5, 16, 32};
        for (int c = 0; c < kHostMaxKc; ++c) {
            const long long b = (!big || c == kHostMaxKc - 1) ? K : (static_cast<long long>(K) * num[c] / den) / 32 * 32;
            if (b > kb[nkc]) kb[++nkc] = b;
            if (!big) break;
        }
        if (nkc == 0) kb[++nkc] = K;  // K == 0: one (empty) chunk
    }
    long long rb[kHostMaxBlk + 1] = {0};
    int nblk = 0;
    {
        const int den = 16, num[kHostMaxBlk] = {10, 13, 15, 16, 16, 16};
        for (int i = 0; i < kHostMaxBlk; ++i) {
            const long long b =
                (!big || i == kHostMaxBlk - 1) ? M : (static_cast<long long>(M) * num[i] / den) / kBM * kBM;
            if (b > rb[nblk]) rb[++nblk] = b;
            if (!big) break;
        }
    }

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
    cudaEvent_t* const ev_done = ev + 3;              // [kHostMaxBlk]: row block's product done
    cudaEvent_t* const ev_in = ev + 3 + kHostMaxBlk;  // [kHostMaxKc]: K chunk's copies in
    // The copy streams start after the workspace exists (stream order of cs).
    bool ok = cudaEventRecord(ev_start, cs) == cudaSuccess &&
              cudaStreamWaitEvent(st->copy_in, ev_start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(st->copy_out, ev_start, 0) == cudaSuccess;

    // Copies in: per K chunk, A's columns (a pitched copy) and B's rows.
    for (int c = 0; c < nkc && ok; ++c) {
        const long long k0 = kb[c], kw = kb[c + 1] - kb[c];
        ok = (kw == 0 ||
              ((K4 == kw && lda == kw
                    ? cudaMemcpyAsync(dA, A, static_cast<size_t>(M) * kw * 4, cudaMemcpyHostToDevice, st->copy_in)
                    : cudaMemcpy2DAsync(dA + k0, static_cast<size_t>(K4) * 4, A + k0, static_cast<size_t>(lda) * 4,
                                        static_cast<size_t>(kw) * 4, static_cast<size_t>(M), cudaMemcpyHostToDevice,
                                        st->copy_in)) == cudaSuccess &&
               copy_rows(dB + k0 * N4, N4, B + k0 * ldb, ldb, kw, N, cudaMemcpyHostToDevice, st->copy_in) ==
                   cudaSuccess)) &&
             cudaEventRecord(ev_in[c], st->copy_in) == cudaSuccess;
    }

    // Products on cs: the chunks before the last over all rows, the last in
    // row blocks; each block's rows of C out on copy_out.
    Scale accumulate;  // C += A_chunk B_chunk for every chunk after the first
    accumulate.alpha = 1.f;
    accumulate.beta = 1.f;
    for (int c = 0; c + 1 < nkc && ok && rc == SGEMM_OK; ++c) {
        ok = cudaStreamWaitEvent(cs, ev_in[c], 0) == cudaSuccess;
        if (ok)
            rc = run_ffma(M, N, static_cast<int>(kb[c + 1] - kb[c]), dA + kb[c], lda_d, dB + kb[c] * N4, ldb_d, dC,
                          ldc_d, stream, nullptr, c > 0 ? &accumulate : nullptr);
    }
    const long long kl0 = kb[nkc - 1], klw = kb[nkc] - kb[nkc - 1];
    if (ok && rc == SGEMM_OK) ok = cudaStreamWaitEvent(cs, ev_in[nkc - 1], 0) == cudaSuccess;
    for (int i = 0; i < nblk && ok && rc == SGEMM_OK; ++i) {
        const long long r0 = rb[i], rows = rb[i + 1] - rb[i];
        rc = run_ffma(static_cast<int>(rows), N, static_cast<int>(klw), dA + r0 * K4 + kl0, lda_d, dB + kl0 * N4,
                      ldb_d, dC + r0 * N4, ldc_d, stream, nullptr, nkc > 1 ? &accumulate : nullptr);
        if (rc != SGEMM_OK) break;
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
