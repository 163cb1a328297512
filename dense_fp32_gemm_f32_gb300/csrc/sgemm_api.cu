// C ABI of the library: argument validation, variant selection, tensor-map
// encoding and launch.  See include/sgemm.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/sgemm.h"
#include "kernels.h"
#include "sgemm_3xtf32_params.h"
#include "sgemm_ffma.cuh"

namespace gb300 {

// Sticky per-device status word; kernels OR error bits into it.
__device__ unsigned int g_sgemm_status = 0;

// Scratch of sgemm_f32_noalloc: room for the stream-K partial tiles and
// ready flags of up to kNoAllocMaxCtas CTAs (10 MiB + 640 bytes), a
// file-scope device array so that the entry point needs no allocation.  Every
// GPU that loads the library holds it until the process exits; all calls on a
// device share it.
constexpr int kNoAllocMaxCtas = 160;
constexpr size_t kNoAllocTileFloats = static_cast<size_t>(kBM) * kBN;  // 128 x 128 tiles only
constexpr size_t kNoAllocFloats = kNoAllocMaxCtas * kNoAllocTileFloats + kNoAllocMaxCtas;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocFloats];

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

// Stream-K scratch kept for one stream (see sk_lease): partial tiles and
// ready flags, allocated once and reused by every call on that stream.
constexpr int kSkCacheEntries = 16;
// Sequence number of calls recorded into a graph: their flags come from a
// fresh workspace zeroed by a memset node, and the counters never hand it out.
constexpr unsigned int kSkSeqCaptured = 0xFFFFFFFFu;
struct SkScratch {
    bool allocated = false;
    unsigned long long stream_id = 0;  // cudaStreamGetId of the stream it serves
    float* ws = nullptr;               // partial tiles
    unsigned int* flags = nullptr;     // one word per CTA
    size_t ws_bytes = 0, nflags = 0;
    unsigned int seq = 0;              // last number handed out
    cudaEvent_t last_use = nullptr;    // recorded on the stream after each call's launch
    int busy = 0;                      // leases not yet returned
    unsigned long long tick = 0;       // last use, for eviction
};

struct DeviceState {
    std::once_flag once;
    int status = SGEMM_ERR_CUDA;  // result of the one-time set-up
    int sm_count = 0;
    int max_clusters_pair = 0;    // co-resident 2-CTA clusters of the FFMA kernel
    int max_clusters_split[9] = {0};
    bool regsplit_ok = false;     // the register-split kernels were built at kRegsLaunch registers
    int fused_per_sm[7] = {0};    // co-resident fused-producer CTAs per SM, by stage count
    unsigned int* status_word = nullptr;  // device address of g_sgemm_status
    std::once_flag pool_once;
    cudaMemPool_t pool = nullptr;  // library-owned pool for per-call workspaces
    std::once_flag noalloc_once;
    int noalloc_status = SGEMM_ERR_CUDA;  // result of looking up g_noalloc_scratch
    float* noalloc_scratch = nullptr;     // its device address on this device
    std::once_flag copy_once;
    cudaStream_t copy_in = nullptr;   // host-buffer entry: host -> device copies
    cudaStream_t copy_out = nullptr;  // host-buffer entry: device -> host copies
    std::mutex sk_mu;                        // guards sk_cache, sk_tick and noalloc_seq
    SkScratch sk_cache[kSkCacheEntries];     // per-stream stream-K scratch (sk_lease)
    unsigned long long sk_tick = 0;
    unsigned int noalloc_seq = 0;            // last sequence number of sgemm_f32_noalloc
};

DeviceState g_dev[kMaxDevices];

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

void load_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            (void)cudaGetLastError();
    });
}

// Largest number of co-resident clusters of `cluster` CTAs (along x or z) for
// one kernel variant; 0 on failure.
int max_active_clusters(const KernelEntry& k, int cx, int cz) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cx, 1, cz);
    cfg.blockDim = dim3(k.threads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(k.smem_bytes);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cx;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = cz;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k.fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

int set_smem_attr(const KernelEntry& k) {
    if (!k.fn) return SGEMM_OK;
    if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem_bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

cudaMemPool_t workspace_pool(int dev, DeviceState& st);

int init_device(int dev, DeviceState& st) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    // The library carries sm_103a code only (compute capability 10.3).
    if (major != 10 || minor != 3) return SGEMM_ERR_UNSUPPORTED;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_sgemm_status) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    st.status_word = static_cast<unsigned int*>(addr);
    st.regsplit_ok = true;
    for (int math = kMathFfma; math <= kMathFfma2; ++math) {
        for (int s = 1; s <= 6; ++s) {
            if (set_smem_attr(ffma_kernel_tma(s, math)) != SGEMM_OK) return SGEMM_ERR_CUDA;
            // setmaxnreg.inc waits until the registers it asks for are free;
            // the split adds up to kRegsLaunch per thread of the CTA, so a
            // kernel built with any other count must never be launched.
            const KernelEntry split_kernels[3] = {ffma_kernel_tma_wg(s, math), ffma_kernel_tma_wide(s, math),
                                                  ffma_kernel_tma_wide_amn(s, math)};
            for (const KernelEntry& wg : split_kernels) {
                if (!wg.fn) {
                    if (&wg == &split_kernels[0]) st.regsplit_ok = false;
                    continue;  // (the wide tile is built for 2..4 stages only)
                }
                if (set_smem_attr(wg) != SGEMM_OK) return SGEMM_ERR_CUDA;
                cudaFuncAttributes fa;
                if (cudaFuncGetAttributes(&fa, wg.fn) != cudaSuccess || fa.numRegs != kRegsLaunch) {
                    (void)cudaGetLastError();
                    st.regsplit_ok = false;
                }
            }
        }
        for (int s = 1; s <= 6; ++s)
            if (set_smem_attr(ffma_kernel_cpasync(s, math)) != SGEMM_OK) return SGEMM_ERR_CUDA;
        for (int v = 0; v < 4; ++v)
            if (set_smem_attr(small_kernel((v & 1) != 0, (v & 2) != 0)) != SGEMM_OK) return SGEMM_ERR_CUDA;
        for (int s = 2; s <= 4; ++s) {
            const KernelEntry f = ffma_kernel_tma_fused(s, math);
            if (set_smem_attr(f) != SGEMM_OK) return SGEMM_ERR_CUDA;
            int n = 0;
            if (f.fn && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f.fn, f.threads,
                                                                      static_cast<size_t>(f.smem_bytes)) != cudaSuccess) {
                (void)cudaGetLastError();
                n = 0;
            }
            if (math == kMathFfma2 || n < st.fused_per_sm[s] || st.fused_per_sm[s] == 0) st.fused_per_sm[s] = n;
        }
        for (int s = 1; s <= 6; ++s) {
            for (int prod : {static_cast<int>(kProducerTma), static_cast<int>(kProducerCpAsync)})
                if (set_smem_attr(ffma_kernel_scaled(prod, s, math)) != SGEMM_OK) return SGEMM_ERR_CUDA;
            for (bool scaled : {false, true}) {
                if (set_smem_attr(ffma_kernel_amn(s, math, scaled)) != SGEMM_OK) return SGEMM_ERR_CUDA;
                if (set_smem_attr(ffma_kernel_tma_x(s, math, scaled)) != SGEMM_OK) return SGEMM_ERR_CUDA;
            }
        }
    }
    if (set_smem_attr(tf32x3_kernel()) != SGEMM_OK || set_smem_attr(tf32x3_direct_kernel()) != SGEMM_OK ||
        set_smem_attr(tf32x3_wide_kernel()) != SGEMM_OK || set_smem_attr(tf32x3_wide_pb_kernel()) != SGEMM_OK)
        return SGEMM_ERR_CUDA;
    const KernelEntry ref = ffma_kernel_tma(4, kMathFfma2);
    st.max_clusters_pair = max_active_clusters(ref, 2, 1);
    st.max_clusters_split[1] = st.sm_count;
    for (int s = 2; s <= 8; ++s) st.max_clusters_split[s] = max_active_clusters(ref, 1, s);
    load_encoder();
    // The pool of per-call workspaces (repack buffers, and the stream-K
    // workspace of calls recorded into a graph) is created here, with the
    // library's first call on the device, so that no call made inside a
    // stream capture has to create it (which the capture would not allow).
    // (Without it, those calls fail; the rest work.)
    (void)workspace_pool(dev, st);
    return SGEMM_OK;
}

// The library's own stream-ordered memory pool on device `dev`, created on
// first use.  Its release threshold keeps freed workspaces cached in the pool
// (the device's default pool would return them to the system at every
// synchronisation and re-allocate on the next call).
cudaMemPool_t workspace_pool(int dev, DeviceState& st) {
    std::call_once(st.pool_once, [&] {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            (void)cudaGetLastError();
            return;
        }
        // Keep up to 256 MiB cached (the stream-K workspaces, ~10-20 MiB, and
        // repack buffers of moderate size); larger repack buffers go back to
        // the system at the next synchronisation.
        uint64_t threshold = 256ull << 20;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &threshold) != cudaSuccess)
            (void)cudaGetLastError();
        st.pool = pool;
    });
    return st.pool;
}

// Per-stream stream-K scratch.  A call on a stream that is not being
// captured borrows the scratch kept for that stream instead of taking a pool
// workspace and zeroing its flags: no allocation and no memset node ahead of
// the kernel (about 3 us per call, measured on GB300).  Each call gets the
// next sequence number of the scratch; a CTA publishes its partial tile by
// storing that number in its flag, and the CTA finishing the tile waits for
// exactly that number, so flags left by earlier calls (smaller numbers) never
// match.  When the counter would reach kSkSeqCaptured the flags are zeroed
// (a memset on the stream) and numbering restarts at 1.  The scratch is keyed
// by the stream's unique id (a destroyed stream's handle can come back for a
// new stream; its id does not).  With more than kSkCacheEntries streams the
// least recently used idle entry moves to the new stream, whose work first
// waits (on the GPU) for the event recorded after the entry's last call.
struct SkLease {
    SkScratch* e = nullptr;
    float* ws = nullptr;
    unsigned int* flags = nullptr;
    unsigned int seq = 0;
};

// Returns SGEMM_OK with a lease, or another status when the scratch cannot be
// used (stream being captured, a failed CUDA call, every entry busy): the
// caller then takes a pool workspace.
int sk_lease(DeviceState& st, cudaStream_t cs, size_t ws_bytes, size_t nflags, SkLease* out) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(cs, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return SGEMM_ERR_UNSUPPORTED;
    unsigned long long id = 0;
    if (cudaStreamGetId(cs, &id) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(st.sk_mu);
    SkScratch* e = nullptr;
    for (SkScratch& c : st.sk_cache)
        if (c.allocated && c.stream_id == id) e = &c;
    if (!e) {
        // An entry never used, else the least recently used idle one.
        for (SkScratch& c : st.sk_cache)
            if (!c.allocated) {
                e = &c;
                break;
            }
        if (!e)
            for (SkScratch& c : st.sk_cache)
                if (c.busy == 0 && (!e || c.tick < e->tick)) e = &c;
        if (!e) return SGEMM_ERR_UNSUPPORTED;
        if (e->allocated) {
            // Another stream's entry: this stream's work waits for its last call.
            if (cudaStreamWaitEvent(cs, e->last_use, 0) != cudaSuccess) {
                (void)cudaGetLastError();
                return SGEMM_ERR_CUDA;
            }
        }
        e->stream_id = id;
    }
    if (!e->allocated || e->ws_bytes < ws_bytes || e->nflags < nflags) {
        // (Re)allocate at the largest size any plan needs on this device.
        if (e->allocated) {
            // Its previous buffers may still be in use by the last call.
            if (cudaEventSynchronize(e->last_use) != cudaSuccess) {
                (void)cudaGetLastError();
                return SGEMM_ERR_CUDA;
            }
            (void)cudaFree(e->ws);
            e->ws = nullptr;
            e->flags = nullptr;
            e->allocated = false;
        }
        if (!e->last_use && cudaEventCreateWithFlags(&e->last_use, cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            e->last_use = nullptr;
            return SGEMM_ERR_CUDA;
        }
        // (one 128 x 256 tile per SM bounds every schedule's partial tiles:
        // one CTA per SM, or two on 128 x 64 tiles)
        const size_t wsb = std::max(ws_bytes, static_cast<size_t>(st.sm_count) * kBM * kBNWide * sizeof(float));
        const size_t nf = std::max(nflags, static_cast<size_t>(2) * st.sm_count);
        void* mem = nullptr;
        if (cudaMalloc(&mem, wsb + nf * sizeof(unsigned int)) != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        e->ws = static_cast<float*>(mem);
        e->flags = reinterpret_cast<unsigned int*>(static_cast<char*>(mem) + wsb);
        e->ws_bytes = wsb;
        e->nflags = nf;
        e->seq = 0;
        e->allocated = true;
        if (cudaMemsetAsync(e->flags, 0, nf * sizeof(unsigned int), cs) != cudaSuccess) {
            (void)cudaGetLastError();
            (void)cudaFree(mem);
            e->allocated = false;
            return SGEMM_ERR_CUDA;
        }
    }
    if (e->seq + 1 == kSkSeqCaptured) {
        if (cudaMemsetAsync(e->flags, 0, e->nflags * sizeof(unsigned int), cs) != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        e->seq = 0;
    }
    e->seq += 1;
    e->busy += 1;
    e->tick = ++st.sk_tick;
    out->e = e;
    out->ws = e->ws;
    out->flags = e->flags;
    out->seq = e->seq;
    return SGEMM_OK;
}

// Ends a lease after the call's launch (launched or not): records the
// entry's last use on the stream.
void sk_return(DeviceState& st, cudaStream_t cs, SkLease& lease) {
    if (!lease.e) return;
    std::lock_guard<std::mutex> lock(st.sk_mu);
    if (cudaEventRecord(lease.e->last_use, cs) != cudaSuccess) (void)cudaGetLastError();
    lease.e->busy -= 1;
    lease.e = nullptr;
}

// Set-up of the current device (once per device per process).
int current_device(int* dev_out, DeviceState** st_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
    // A host thread whose only CUDA calls so far were queries like the one
    // above has no current context, which the driver calls of the library
    // (tensor-map encoding) need: bind the device's primary context, once per
    // thread and device.
    thread_local uint64_t bound = 0;
    if (!(bound & (uint64_t{1} << dev))) {
        if (cudaSetDevice(dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        bound |= uint64_t{1} << dev;
    }
    DeviceState& st = g_dev[dev];
    std::call_once(st.once, [&] { st.status = init_device(dev, st); });
    *dev_out = dev;
    *st_out = &st;
    return st.status;
}

bool ranges_overlap(const void* a, size_t abytes, const void* b, size_t bbytes) {
    if (!abytes || !bbytes) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

size_t span_bytes(long long rows, long long cols, long long ld) {
    if (rows <= 0 || cols <= 0) return 0;
    return static_cast<size_t>(((rows - 1) * ld + cols) * 4);
}

// a_mn: A is stored transposed (K x M, lda >= M).
int validate(int M, int N, int K, const float* A, int lda, const float* B, int ldb, const float* C, int ldc,
             bool a_mn = false) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (lda < (a_mn ? M : K) || ldb < N || ldc < N) return SGEMM_ERR_INVALID_ARG;
    if (M > 0 && K > 0 && !A) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && N > 0 && !B) return SGEMM_ERR_INVALID_ARG;
    if (M > 0 && N > 0 && !C) return SGEMM_ERR_INVALID_ARG;
    // Output tiles are numbered with a 32-bit int.
    if (((static_cast<long long>(M) + kBM - 1) / kBM) * (((static_cast<long long>(N) + kBN - 1) / kBN) + 1) >
        0x7fffffffLL)
        return SGEMM_ERR_INVALID_ARG;
    const size_t cb = span_bytes(M, N, ldc);
    if (ranges_overlap(C, cb, A, a_mn ? span_bytes(K, M, lda) : span_bytes(M, K, lda)) ||
        ranges_overlap(C, cb, B, span_bytes(K, N, ldb)))
        return SGEMM_ERR_INVALID_ARG;
    return SGEMM_OK;
}

// Operands copied into 16-byte pitched rows (see pack_rows) for the length of
// one call: the copies come from the library's pool and go back to it, in
// stream order, by release().
struct Repacked {
    void* ws = nullptr;
    cudaStream_t stream = nullptr;

    // Copies operand A (mask bit 0) and/or B (bit 1) and points A / lda and
    // B / ldb at the copies, which are always the plain (untransposed) M x K
    // and K x N operands: with transa, A is stored K x M and its copy is the
    // transpose; with transb, likewise B (stored N x K).  SGEMM_ERR_CUDA if
    // the pool cannot serve them (nothing is enqueued then).
    int make(int dev, DeviceState& st, int mask, int M, int N, int K, const float*& A, int& lda, const float*& B,
             int& ldb, cudaStream_t cs, bool transa = false, bool transb = false) {
        stream = cs;
        const long long K4 = (static_cast<long long>(K) + 3) / 4 * 4;
        const long long N4 = (static_cast<long long>(N) + 3) / 4 * 4;
        if (K4 > 0x7fffffffLL || N4 > 0x7fffffffLL) return SGEMM_ERR_INVALID_ARG;
        const size_t bytes_a = (mask & 1) ? ((static_cast<size_t>(M) * K4 * 4 + 255) & ~size_t{255}) : 0;
        const size_t bytes_b = (mask & 2) ? static_cast<size_t>(K) * N4 * 4 : 0;
        cudaMemPool_t pool = workspace_pool(dev, st);
        if (!pool || cudaMallocFromPoolAsync(&ws, bytes_a + bytes_b, pool, cs) != cudaSuccess) {
            (void)cudaGetLastError();
            ws = nullptr;
            return SGEMM_ERR_CUDA;
        }
        float* Ap = (mask & 1) ? static_cast<float*>(ws) : nullptr;
        float* Bp = (mask & 2) ? reinterpret_cast<float*>(static_cast<char*>(ws) + bytes_a) : nullptr;
        // Row copies in one launch, transposing copies in another.
        int rc = pack_rows(A, lda, transa ? nullptr : Ap, K4, M, K, B, ldb, transb ? nullptr : Bp, N4, K, N, cs);
        if (rc == SGEMM_OK)
            rc = transpose_rows(A, lda, transa ? Ap : nullptr, K4, M, K, B, ldb, transb ? Bp : nullptr, N4, K, N, cs);
        if (rc != SGEMM_OK) {
            release();
            return rc;
        }
        if (Ap) {
            A = Ap;
            lda = static_cast<int>(K4);
        }
        if (Bp) {
            B = Bp;
            ldb = static_cast<int>(N4);
        }
        return SGEMM_OK;
    }
    // A (M x K, pitch lda) -> its transpose (K x M, pitch M rounded up to 4
    // floats) in a pool buffer; A / lda then point at the copy.
    int make_transposed_a(int dev, DeviceState& st, int M, int K, const float*& A, int& lda, cudaStream_t cs) {
        stream = cs;
        const long long M4 = (static_cast<long long>(M) + 3) / 4 * 4;
        if (M4 > 0x7fffffffLL) return SGEMM_ERR_INVALID_ARG;
        cudaMemPool_t pool = workspace_pool(dev, st);
        if (!pool || cudaMallocFromPoolAsync(&ws, static_cast<size_t>(K) * M4 * 4, pool, cs) != cudaSuccess) {
            (void)cudaGetLastError();
            ws = nullptr;
            return SGEMM_ERR_CUDA;
        }
        float* At = static_cast<float*>(ws);
        const int rc = transpose_rows(A, lda, At, M4, K, M, nullptr, 0, nullptr, 0, 0, 0, cs);
        if (rc != SGEMM_OK) {
            release();
            return rc;
        }
        A = At;
        lda = static_cast<int>(M4);
        return SGEMM_OK;
    }
    void release() {
        if (ws) (void)cudaFreeAsync(ws, stream);
        ws = nullptr;
    }
};

// A read in the transposed layout: the consumers read each k's A values as
// two 16-byte vectors instead of a 4-k vector per row (82 -> 89 % FMA-pipe
// duty).  Two ways to get there: a transposing copy of A in HBM
// (sgemm_options.a_layout = 2; the transposed-A kernels, no extra work in
// the kernel) or two producer warps transposing each A slice in shared
// memory (SGEMM_PRODUCER_TMA_X; no copy, a little more shared-memory traffic
// in the kernel).  Measured on GB300 (TFLOP/s, A read as stored / copy in HBM
// / transposed in shared memory): 2048^3 62.0 / 62.7 / 66.9, 4096^3 65.4 /
// 68.5 / 70.5, 8192^3 66.4 / 71.2 / 71.0, 128 x 8192 x 16384 64.2 / 68.2 /
// 68.7, 8192 x 128 x 8192 62.0 / - / 66.4.  The copy costs one read and one
// write of A (~1/N of the product) and a pool buffer of A's size; with the
// two transposing warps it no longer wins anywhere, so it is taken only when
// forced (a_layout = 2) and the transposition in shared memory is automatic
// (make_plan).  (The general entry's A stored transposed is read in place by
// the transposed-A kernels: no copy.)

bool options_force_variant(const sgemm_options* opt) {
    return opt && (opt->producer || opt->split_k || opt->multicast || opt->math || opt->stages || opt->tail_split ||
                   opt->stream_k || opt->tile_n || opt->repack);
}

// 0 = keep A as stored, 1 = copy it transposed; -1 = invalid option.
int choose_a_layout(int K, const sgemm_options* opt) {
    const int want = opt ? opt->a_layout : 0;
    if (want < 0 || want > 2) return -1;
    return (K > 0 && want == 2) ? 1 : 0;
}

struct Launch {
    int tile_base = 0;  // first output tile
    int tiles = 0;      // output tiles in this launch (grid x)
    int split = 1;      // CTAs per tile along K (cluster z)
};

struct Plan {
    int producer = kProducerTma;
    int math = kMathFfma2;
    int stages = 4;
    int mcast = 1;
    int bn = kBN;     // output tile width (kBN or kBNWide)
    int tiles_n = 0;  // tiles per row of tiles (padded to even for multicast pairs)
    int num_k_tiles = 0;
    int nlaunch = 1;
    Launch launch[2];
    int sk = 0;           // stream-K: launch[0].tiles CTAs, one per SM
    int sk_dp_tiles = 0;  // tiles taken whole (data-parallel waves) before the stream-K region
    int repack = 0;       // operands copied to 16-byte pitched rows first: bit 0 = A, bit 1 = B
    bool a_mn = false;    // A stored transposed (K x M): the transposed-A kernels
};

// Repacking pays once the product is large next to the copy.  Measured on
// GB300 (both operands misaligned, one copy launch for both): 1023 x 1025 x
// 1027 (2^31 flop) 65 us against 69 us with cp.async, 2047 x 2049 x 2051
// +23 %, 4095 x 4097 x 4099 and 8191 x 8193 x 8195 +30 %.
constexpr double kRepackMinFlops = 1073741824.0;  // 2^30

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

bool is_tma(int producer) {
    return producer == kProducerTma || producer == kProducerTmaWg || producer == kProducerFused ||
           producer == kProducerTmaX;
}

KernelEntry ffma_kernel(const Plan& pl) {
    if (pl.a_mn) return pl.producer == kProducerTma     ? ffma_kernel_amn(pl.stages, pl.math, false)
                        : pl.producer == kProducerTmaWg ? ffma_kernel_tma_wide_amn(pl.stages, pl.math)
                                                        : KernelEntry{nullptr, 0, 0};
    if (pl.producer == kProducerFused) return ffma_kernel_tma_fused(pl.stages, pl.math);
    if (pl.producer == kProducerTmaX) return ffma_kernel_tma_x(pl.stages, pl.math, false);
    if (pl.bn == kBNWide) return pl.producer == kProducerTmaWg ? ffma_kernel_tma_wide(pl.stages, pl.math)
                                                                : KernelEntry{nullptr, 0, 0};
    switch (pl.producer) {
        case kProducerTma: return ffma_kernel_tma(pl.stages, pl.math);
        case kProducerTmaWg: return ffma_kernel_tma_wg(pl.stages, pl.math);
        case kProducerCpAsync: return ffma_kernel_cpasync(pl.stages, pl.math);
    }
    return {nullptr, 0, 0};
}

const char* producer_name(int producer) {
    switch (producer) {
        case kProducerTma: return "tma";
        case kProducerTmaWg: return "tmawg";
        case kProducerFused: return "fused";
        case kProducerTmaX: return "tmax";
        case kProducerCpAsync: return "cpasync";
    }
    return "?";
}

bool tma_ok(const float* p, int ld) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (static_cast<long long>(ld) * 4) % 16 == 0;
}

// Chooses the variant.  Any field of `opt` that is non-zero forces that choice.
int make_plan(const DeviceState& st, int M, int N, int K, const float* A, int lda, const float* B, int ldb,
              const sgemm_options* opt, Plan* out, bool a_mn = false) {
    Plan pl;
    // Transposed A (general entry only): tensor-map readable A, TMA producer
    // warp, 2 stages, paired FMA, no multicast (see below).
    if (a_mn && (K == 0 || !tma_ok(A, lda) ||
                 (opt && (opt->producer || (opt->tile_n && opt->tile_n != kBNWide) || opt->math || opt->stages ||
                          opt->multicast == 2))))
        return SGEMM_ERR_INVALID_ARG;
    pl.a_mn = a_mn;
    pl.num_k_tiles = static_cast<int>(ceil_div(K, kBK));
    long long tiles_n = ceil_div(N, kBN);
    const long long tiles_m = ceil_div(M, kBM);

    // Producer: tensor maps need 16-byte aligned bases and row strides, and
    // K > 0.  An operand without them is either repacked into pitched rows
    // (which the tensor maps can address) or read by the cp.async producer.
    const int want_prod = opt ? opt->producer : 0;
    const int want_repack = opt ? opt->repack : 0;
    if (want_repack < 0 || want_repack > 2) return SGEMM_ERR_INVALID_ARG;
    const int misaligned = (a_mn || tma_ok(A, lda) ? 0 : 1) | (tma_ok(B, ldb) ? 0 : 2);
    if (K > 0 && misaligned &&
        (want_repack == 2 || a_mn ||  // (the transposed-A kernels have no cp.async form)
         (want_repack == 0 && want_prod == SGEMM_PRODUCER_AUTO &&
          2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) >= kRepackMinFlops)))
        pl.repack = misaligned;
    const bool aligned = K > 0 && (misaligned & ~pl.repack) == 0;
    if (want_prod == SGEMM_PRODUCER_TMA) {
        if (!aligned) return SGEMM_ERR_INVALID_ARG;
        pl.producer = kProducerTma;
    } else if (want_prod == SGEMM_PRODUCER_TMA_WG) {
        if (!aligned) return SGEMM_ERR_INVALID_ARG;
        if (!st.regsplit_ok) return SGEMM_ERR_UNSUPPORTED;
        pl.producer = kProducerTmaWg;
    } else if (want_prod == SGEMM_PRODUCER_TMA_X) {
        if (!aligned || a_mn) return SGEMM_ERR_INVALID_ARG;
        pl.producer = kProducerTmaX;
    } else if (want_prod == SGEMM_PRODUCER_FUSED) {
        if (!aligned) return SGEMM_ERR_INVALID_ARG;
        pl.producer = kProducerFused;
    } else if (want_prod == SGEMM_PRODUCER_CPASYNC) {
        pl.producer = kProducerCpAsync;
    } else if (want_prod == SGEMM_PRODUCER_AUTO) {
        // Tensor maps: A transposed in shared memory, unless it already is in
        // HBM (a_mn) or another choice rules the transposing warps out.
        const bool x_ok = !a_mn && !(opt && (opt->multicast == 2 || (opt->tile_n && opt->tile_n != kBN) ||
                                             (opt->stages && (opt->stages < 2 || opt->stages > 4))));
        pl.producer = !aligned ? kProducerCpAsync : x_ok ? kProducerTmaX : kProducerTma;
    } else {
        return SGEMM_ERR_INVALID_ARG;
    }

    // Tile width: 128 x 256 tiles need the producer warpgroup (register
    // split) and so tensor maps.
    const int want_bn = opt ? opt->tile_n : 0;
    if (want_bn == kBNWide) {
        if (want_prod == SGEMM_PRODUCER_AUTO) {
            if (!aligned) return SGEMM_ERR_INVALID_ARG;
            if (!st.regsplit_ok) return SGEMM_ERR_UNSUPPORTED;
            pl.producer = kProducerTmaWg;
        }
        if (pl.producer != kProducerTmaWg) return SGEMM_ERR_INVALID_ARG;
        pl.bn = kBNWide;
    } else if (want_bn == kBNFused) {
        // 128 x 64 tiles: the fused-producer CTAs, two per SM.
        if (want_prod == SGEMM_PRODUCER_AUTO) {
            if (!aligned) return SGEMM_ERR_INVALID_ARG;
            pl.producer = kProducerFused;
        }
        if (pl.producer != kProducerFused) return SGEMM_ERR_INVALID_ARG;
    } else if (want_bn != 0 && want_bn != kBN) {
        return SGEMM_ERR_INVALID_ARG;
    }
    if (pl.producer == kProducerFused) pl.bn = kBNFused;

    if (opt && opt->math) {
        if (opt->math != kMathFfma && opt->math != kMathFfma2) return SGEMM_ERR_INVALID_ARG;
        pl.math = opt->math;
    }
    // Stages: two for the tensor-map producers (measured on GB300 with the
    // paired-FMA consumers: 0.3-2 % faster than 3-6 at every named problem,
    // 20-25 % faster than one), four for cp.async, whose 4-byte copies have
    // more latency to hide.
    pl.stages = pl.producer == kProducerCpAsync ? 4 : 2;
    if (opt && opt->stages) {
        if (opt->stages < 1 || opt->stages > 6) return SGEMM_ERR_INVALID_ARG;
        pl.stages = opt->stages;
    }
    if (pl.producer == kProducerCpAsync && pl.stages != 2 && pl.stages != 4) {
        if (opt && opt->stages) return SGEMM_ERR_INVALID_ARG;
        pl.stages = 4;
    }
    if (pl.producer == kProducerFused && !(opt && opt->stages)) pl.stages = 4;
    if ((pl.bn == kBNWide || pl.bn == kBNFused || pl.producer == kProducerTmaX) && (pl.stages < 2 || pl.stages > 4))
        return SGEMM_ERR_INVALID_ARG;
    if (pl.producer == kProducerTmaX && pl.bn != kBN) return SGEMM_ERR_INVALID_ARG;
    // CTAs that can be resident at once, for the stream-K grid.
    const int per_sm = pl.producer == kProducerFused ? st.fused_per_sm[pl.stages] : 1;
    if (per_sm < 1) return SGEMM_ERR_UNSUPPORTED;
    const long long slots = static_cast<long long>(st.sm_count) * per_sm;

    tiles_n = ceil_div(N, pl.bn);
    const long long tiles = tiles_n * tiles_m;

    // Stream-K (decided first; see below for the schedule).  Automatic
    // whenever nothing else is forced and there are at least two (tile, K
    // slice) units per SM: measured on GB300 it beats the plain grid and
    // cluster split-K (1024^3 +8 %, 2048^3 +16 %, 4096^3 +4 %, 8192^3 +1 %,
    // 8192x128x8192 +22 %); tiny problems keep cluster split-K.
    const int want_sk = opt ? opt->stream_k : 0;
    if (want_sk < 0 || want_sk > 2) return SGEMM_ERR_INVALID_ARG;
    const bool forced_other = opt && (opt->split_k || opt->multicast == 2 || opt->tail_split > 1);
    const bool use_sk = want_sk == 2 || (want_sk == 0 && !forced_other && pl.num_k_tiles > 0 &&
                                         tiles * pl.num_k_tiles >= 2LL * slots);

    // Split-K over the whole grid, only when the tiles do not fill one wave:
    // pick s in 1..8 minimising (waves of clusters) x (K tiles per CTA).  (With
    // a wave or more, only the last partial wave is split; see below.)
    int split = 1;
    if (opt && opt->split_k) {
        if (opt->split_k < 1 || opt->split_k > 8) return SGEMM_ERR_INVALID_ARG;
        split = opt->split_k;
    } else if (tiles < st.sm_count && !use_sk && pl.producer != kProducerFused) {
        long long best = -1;
        for (int s = 1; s <= 8; ++s) {
            const int slots = st.max_clusters_split[s];
            if (slots <= 0) continue;
            if (s > 1 && pl.num_k_tiles < 2 * s) break;  // keep at least two K slices per CTA
            const long long cost = ceil_div(tiles, slots) * ceil_div(pl.num_k_tiles, s);
            if (best < 0 || cost < best) {
                best = cost;
                split = s;
            }
        }
    }
    if (split > 1 && pl.stages < 2) return SGEMM_ERR_INVALID_ARG;  // partial tile needs 64 KiB of ring
    if (split > 1 && pl.producer == kProducerFused) return SGEMM_ERR_INVALID_ARG;  // two CTAs per SM: no clusters

    // Multicast pairs along N (TMA producer, no split).  Measured on GB300 at
    // 1024^3..8192^3 the pairing costs more (the two CTAs release every slot
    // in lock step) than the halved L2->SM traffic for A saves, so it is off
    // unless forced.
    const int want_mc = opt ? opt->multicast : 0;
    if (want_mc == 2) {
        if (split > 1 || !is_tma(pl.producer) || pl.producer == kProducerFused || pl.producer == kProducerTmaX)
            return SGEMM_ERR_INVALID_ARG;
        if (st.max_clusters_pair < 1) return SGEMM_ERR_UNSUPPORTED;
        pl.mcast = 2;
    } else if (want_mc == 0 || want_mc == 1) {
        pl.mcast = 1;
    } else {
        return SGEMM_ERR_INVALID_ARG;
    }
    pl.tiles_n = static_cast<int>(pl.mcast == 2 ? 2 * ceil_div(tiles_n, 2) : tiles_n);
    const long long grid_tiles = static_cast<long long>(pl.tiles_n) * tiles_m;

    // Last partial wave.  When the tiles do not fill a whole number of waves,
    // the last wave leaves SMs idle for a full tile time.  Those tiles can run
    // as a second launch split along K (clusters + shared-memory reduction),
    // so that more CTAs share the tail at 1/s of the work each; the modelled
    // tail time, in full-K tile times, is ceil(rem / clusters_s) / s.  On
    // GB300 the measured tail is well above that model (4096^3: 112 tail tiles
    // split 5 ways made the call 3 % slower; 2048^3: 104 tiles split 4 ways,
    // 2.6 % faster), so it is taken only when forced (tail_split = 2..8).
    pl.nlaunch = 1;
    pl.launch[0].tile_base = 0;
    pl.launch[0].tiles = static_cast<int>(grid_tiles);
    pl.launch[0].split = split;
    const int want_tail = opt ? opt->tail_split : 0;
    if (want_tail < 0 || want_tail > 8) return SGEMM_ERR_INVALID_ARG;
    if (split == 1 && pl.mcast == 1 && want_tail > 1 && grid_tiles > st.sm_count && pl.producer != kProducerFused) {
        const long long full = (grid_tiles / st.sm_count) * st.sm_count;
        const long long rem = grid_tiles - full;
        // keep at least four K slices per CTA of the tail
        if (rem > 0 && st.max_clusters_split[want_tail] > 0 && pl.num_k_tiles >= 4 * want_tail) {
            pl.nlaunch = 2;
            pl.launch[0].tiles = static_cast<int>(full);
            pl.launch[1].tile_base = static_cast<int>(full);
            pl.launch[1].tiles = static_cast<int>(rem);
            pl.launch[1].split = want_tail;
        }
    }

    // Stream-K schedule: one CTA per SM (two for the fused producer), partial
    // tiles finished through a global workspace.
    if (use_sk) {
        if (split > 1 || pl.mcast > 1 || pl.nlaunch > 1 || pl.num_k_tiles == 0) return SGEMM_ERR_INVALID_ARG;
        // All but the last full wave run data-parallel (raster order keeps
        // the A and B panels in flight few, as in the plain launch); the last
        // full wave and the partial one are dealt out as units.
        const long long G = slots;
        const long long waves = grid_tiles / G;
        const long long dp = waves > 1 ? (waves - 1) * G : 0;
        const long long units = (grid_tiles - dp) * pl.num_k_tiles;
        pl.sk = 1;
        pl.sk_dp_tiles = static_cast<int>(dp);
        pl.nlaunch = 1;
        pl.launch[0].tile_base = 0;
        pl.launch[0].split = 1;
        pl.launch[0].tiles = static_cast<int>(units < G ? units : G);
    }
    *out = pl;
    return SGEMM_OK;
}

int encode_2d(CUtensorMap* map, const float* base, long long inner, long long outer, long long ld, int box_inner,
              int box_outer, CUtensorMapSwizzle swz) {
    if (!g_encode) return SGEMM_ERR_UNSUPPORTED;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGEMM_OK : SGEMM_ERR_CUDA;
}

const char* describe_plan(const Plan& pl) {
    static thread_local char buf[128];
    int n = std::snprintf(buf, sizeof buf, "%s/%s/mc%d/s%d/st%d", producer_name(pl.producer),
                          pl.math == kMathFfma2 ? "ffma2" : "ffma", pl.mcast, pl.launch[0].split, pl.stages);
    if (pl.nlaunch > 1 && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/tail%d:%d", pl.launch[1].split, pl.launch[1].tiles);
    if (pl.sk && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/sk%d", pl.launch[0].tiles);
    if (pl.bn != kBN && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/n%d", pl.bn);
    if (pl.repack && n > 0 && n < static_cast<int>(sizeof buf))
        n += std::snprintf(buf + n, sizeof buf - n, "/repack%s", pl.repack == 1 ? "A" : pl.repack == 2 ? "B" : "AB");
    if (pl.a_mn && n > 0 && n < static_cast<int>(sizeof buf))
        std::snprintf(buf + n, sizeof buf - n, "/at");
    return buf;
}

// Epilogue scaling of the general entry: C = alpha * A B + beta * C.
struct Scale {
    float alpha = 1.f, beta = 0.f;
};

// Small problems: the 32 x 32-tile kernel when the 128 x 128 tiles would be
// too few to occupy the GPU and the product is small (see small_problem).
constexpr double kSmallMaxFlops = 268435456.0;  // 2^28

bool small_problem(const DeviceState& st, int M, int N, int K) {
    const long long tiles = ceil_div(M, kBM) * ceil_div(N, kBN);
    return 2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) <= kSmallMaxFlops &&
           4 * tiles <= st.sm_count;
}

// A forced small kernel takes no other forced choice (it has no producer,
// stages, split or tile options, and no waits for debug_skip_stage to time out).
bool small_forced_ok(const sgemm_options* opt) {
    return !(opt->split_k || opt->multicast || opt->math || opt->stages || opt->tail_split || opt->stream_k ||
             opt->tile_n || opt->repack || opt->a_layout || opt->debug_skip_stage);
}

int launch_small(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                 void* stream, const Scale* scale, bool a_mn) {
    const bool scaled = scale && (scale->alpha != 1.f || scale->beta != 0.f);
    const KernelEntry k = small_kernel(a_mn, scaled);
    SmallParams prm;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.A = A;
    prm.lda = lda;
    prm.B = B;
    prm.ldb = ldb;
    prm.C = C;
    prm.ldc = ldc;
    prm.alpha = scale ? scale->alpha : 1.f;
    prm.beta = scale ? scale->beta : 0.f;
    const long long gx = ceil_div(N, kSmallTile), gy = ceil_div(M, kSmallTile);
    if (gy > 65535) return SGEMM_ERR_INVALID_ARG;  // (never: the rule and the forced form both bound M)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
    cfg.blockDim = dim3(k.threads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(k.smem_bytes);
    cfg.stream = static_cast<cudaStream_t>(stream);
    void* args[1] = {&prm};
    if (cudaLaunchKernelExC(&cfg, k.fn, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

int run_ffma(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
             void* stream, const sgemm_options* opt, const Scale* scale = nullptr, bool a_mn = false) {
    int rc = validate(M, N, K, A, lda, B, ldb, C, ldc, a_mn);
    if (rc != SGEMM_OK) return rc;
    if (opt && opt->debug_skip_stage < 0) return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;  // nothing to write; no device work
    int dev = 0;
    DeviceState* st = nullptr;
    rc = current_device(&dev, &st);
    if (rc != SGEMM_OK) return rc;

    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (opt && opt->producer == SGEMM_PRODUCER_SMALL) {
        if (!small_forced_ok(opt)) return SGEMM_ERR_INVALID_ARG;
        if (ceil_div(M, kSmallTile) > 65535) return SGEMM_ERR_INVALID_ARG;
        return launch_small(M, N, K, A, lda, B, ldb, C, ldc, stream, scale, a_mn);
    }
    if (!options_force_variant(opt) && !(opt && (opt->a_layout || opt->debug_skip_stage)) &&
        small_problem(*st, M, N, K))
        return launch_small(M, N, K, A, lda, B, ldb, C, ldc, stream, scale, a_mn);
    // A copied transposed for the transposed-A kernels (see choose_a_layout).
    Repacked a_t;
    const int layout = a_mn ? 0 : choose_a_layout(K, opt);
    if (layout < 0) return SGEMM_ERR_INVALID_ARG;
    if (layout == 1) {
        rc = a_t.make_transposed_a(dev, *st, M, K, A, lda, cs);
        if (rc == SGEMM_OK) {
            a_mn = true;
        } else if (opt && opt->a_layout == 2) {
            return rc;
        }  // (automatic: without the pool's buffer, A is read as stored)
    }
    // (With a transposed A, make_plan rejects forced producer, tile, math,
    // stage and multicast choices: the transposed-A kernels have one form.)
    Plan pl;
    rc = make_plan(*st, M, N, K, A, lda, B, ldb, opt, &pl, a_mn);
    if (rc != SGEMM_OK) {
        a_t.release();
        return rc;
    }

    // Repacking: copy the misaligned operand(s) into pitched rows taken from
    // the pool, and run the product on the copies.  If the pool cannot serve
    // the copies, the automatic choice falls back to the cp.async producer.
    Repacked packed;
    if (pl.repack) {
        rc = packed.make(dev, *st, pl.repack, M, N, K, A, lda, B, ldb, cs);
        if (rc == SGEMM_ERR_CUDA && !(opt && opt->repack == 2)) {
            sgemm_options o = opt ? *opt : sgemm_options{};
            o.repack = 1;
            rc = make_plan(*st, M, N, K, A, lda, B, ldb, &o, &pl, a_mn);
        }
        if (rc != SGEMM_OK) {
            a_t.release();
            return rc;
        }
    }
    // Returns the copies of A and B to the pool behind everything enqueued so far.
    auto release_pack = [&] {
        packed.release();
        a_t.release();
    };

    const bool scaled = scale && (scale->alpha != 1.f || scale->beta != 0.f);
    const KernelEntry k = pl.a_mn ? (pl.bn == kBN ? ffma_kernel_amn(pl.stages, pl.math, scaled)
                                                  : scaled ? KernelEntry{nullptr, 0, 0} : ffma_kernel(pl))
                          : scaled ? (pl.producer == kProducerTmaX ? ffma_kernel_tma_x(pl.stages, pl.math, true)
                                      : pl.bn == kBN               ? ffma_kernel_scaled(pl.producer, pl.stages, pl.math)
                                                                   : KernelEntry{nullptr, 0, 0})
                                   : ffma_kernel(pl);
    if (!k.fn) {
        release_pack();
        return SGEMM_ERR_INVALID_ARG;
    }

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    std::memset(&tmA, 0, sizeof tmA);
    std::memset(&tmB, 0, sizeof tmB);
    if (is_tma(pl.producer)) {
        rc = pl.a_mn ? encode_2d(&tmA, A, M, K, lda, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_NONE)  // {m, k} boxes of 128 x 32
                     : encode_2d(&tmA, A, K, M, lda, kBK, kBM / pl.mcast, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc == SGEMM_OK) rc = encode_2d(&tmB, B, N, K, ldb, pl.bn, kBK, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != SGEMM_OK) {
            release_pack();
            return rc;
        }
    }

    FfmaParams prm;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.A = A;
    prm.lda = lda;
    prm.B = B;
    prm.ldb = ldb;
    prm.C = C;
    prm.ldc = ldc;
    prm.num_k_tiles = pl.num_k_tiles;
    prm.mcast = pl.mcast;
    prm.vec_store = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0) ? 1 : 0;
    prm.tiles_n = pl.tiles_n;
    prm.skip_stage = opt ? opt->debug_skip_stage : 0;
    prm.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
    prm.status = st->status_word;
    prm.alpha = scale ? scale->alpha : 1.f;
    prm.beta = scale ? scale->beta : 0.f;
    prm.sk = pl.sk;
    prm.sk_dp_tiles = pl.sk_dp_tiles;
    prm.sk_units = (static_cast<long long>(pl.tiles_n) * ceil_div(M, kBM) - pl.sk_dp_tiles) * pl.num_k_tiles;
    prm.ws = nullptr;
    prm.flags = nullptr;
    prm.sk_seq = kSkSeqCaptured;

    // Stream-K workspace: one partial tile and one flag per CTA, from the
    // stream's own scratch (sk_lease) or, while the stream is being captured
    // into a graph, from the library's stream-ordered pool for this call with
    // its flags zeroed by a memset (stream order makes concurrent calls on
    // different streams use different workspaces).
    void* ws = nullptr;
    SkLease lease;
    if (pl.sk) {
        const size_t G = static_cast<size_t>(pl.launch[0].tiles);
        const size_t tile_bytes = static_cast<size_t>(kBM) * pl.bn * sizeof(float);
        if (sk_lease(*st, cs, G * tile_bytes, G, &lease) == SGEMM_OK) {
            prm.ws = lease.ws;
            prm.flags = lease.flags;
            prm.sk_seq = lease.seq;
        } else {
            cudaMemPool_t pool = workspace_pool(dev, *st);
            if (!pool ||
                cudaMallocFromPoolAsync(&ws, G * tile_bytes + G * sizeof(unsigned int), pool, cs) != cudaSuccess) {
                (void)cudaGetLastError();
                release_pack();
                return SGEMM_ERR_CUDA;
            }
            prm.ws = static_cast<float*>(ws);
            prm.flags = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + G * tile_bytes);
            if (cudaMemsetAsync(prm.flags, 0, G * sizeof(unsigned int), cs) != cudaSuccess) {
                (void)cudaGetLastError();
                (void)cudaFreeAsync(ws, cs);
                release_pack();
                return SGEMM_ERR_CUDA;
            }
        }
    }

    for (int l = 0; l < pl.nlaunch; ++l) {
        const Launch& ln = pl.launch[l];
        if (ln.tiles <= 0) continue;
        prm.tile_base = ln.tile_base;
        prm.split = ln.split;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ln.tiles), 1, static_cast<unsigned>(ln.split));
        cfg.blockDim = dim3(k.threads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(k.smem_bytes);
        cfg.stream = static_cast<cudaStream_t>(stream);
        cudaLaunchAttribute attr;
        if (pl.sk) {
            // Finishing CTAs wait for the partial tiles of later CTAs: all of
            // them must be resident at once.
            attr.id = cudaLaunchAttributeCooperative;
            attr.val.cooperative = 1;
        } else {
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = pl.mcast;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = ln.split;
        }
        cfg.attrs = &attr;
        cfg.numAttrs = (pl.sk || pl.mcast > 1 || ln.split > 1) ? 1 : 0;
        void* args[3] = {&tmA, &tmB, &prm};
        if (cudaLaunchKernelExC(&cfg, k.fn, args) != cudaSuccess) {
            (void)cudaGetLastError();
            sk_return(*st, cs, lease);
            if (ws) (void)cudaFreeAsync(ws, cs);
            release_pack();
            return SGEMM_ERR_CUDA;
        }
    }
    sk_return(*st, cs, lease);
    release_pack();
    if (ws && cudaFreeAsync(ws, cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

// sgemm_f32 with the stream-K workspace in g_noalloc_scratch instead of a
// pool allocation (see sgemm_f32_noalloc in include/sgemm.h).
int run_ffma_noalloc(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                     void* stream) {
    int rc = validate(M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    int dev = 0;
    DeviceState* st = nullptr;
    rc = current_device(&dev, &st);
    if (rc != SGEMM_OK) return rc;
    // Set-up, once per device with that device current: the host-side name
    // g_noalloc_scratch is only a stand-in; the kernel needs the array's
    // device address.
    std::call_once(st->noalloc_once, [&] {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) {
            (void)cudaGetLastError();
            st->noalloc_status = SGEMM_ERR_CUDA;
            return;
        }
        st->noalloc_scratch = static_cast<float*>(addr);
        st->noalloc_status = SGEMM_OK;
    });
    if (st->noalloc_status != SGEMM_OK) return st->noalloc_status;
    if (small_problem(*st, M, N, K)) return launch_small(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr, false);

    // Plan: stream-K whenever there is a K slice to deal out (K == 0 runs the
    // plain grid, which writes zeros and needs no scratch).
    sgemm_options o = {};
    o.stream_k = K > 0 ? 2 : 1;
    o.split_k = K > 0 ? 0 : 1;
    o.tile_n = kBN;
    o.repack = 1;  // repacking would allocate: misaligned operands take the cp.async producer
    Plan pl;
    rc = make_plan(*st, M, N, K, A, lda, B, ldb, &o, &pl);
    if (rc != SGEMM_OK) return rc;
    if (pl.sk && pl.launch[0].tiles > kNoAllocMaxCtas) pl.launch[0].tiles = kNoAllocMaxCtas;
    const size_t G = pl.sk ? static_cast<size_t>(pl.launch[0].tiles) : 0;
    if (G * kBM * pl.bn + G > kNoAllocFloats) return SGEMM_ERR_INVALID_ARG;  // cannot happen with the cap

    const KernelEntry k = ffma_kernel(pl);
    if (!k.fn) return SGEMM_ERR_INVALID_ARG;
    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    std::memset(&tmA, 0, sizeof tmA);
    std::memset(&tmB, 0, sizeof tmB);
    if (is_tma(pl.producer)) {
        rc = encode_2d(&tmA, A, K, M, lda, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc == SGEMM_OK) rc = encode_2d(&tmB, B, N, K, ldb, pl.bn, kBK, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != SGEMM_OK) return rc;
    }

    FfmaParams prm;
    std::memset(&prm, 0, sizeof prm);
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.A = A;
    prm.lda = lda;
    prm.B = B;
    prm.ldb = ldb;
    prm.C = C;
    prm.ldc = ldc;
    prm.num_k_tiles = pl.num_k_tiles;
    prm.split = 1;
    prm.mcast = 1;
    prm.vec_store = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0) ? 1 : 0;
    prm.tile_base = 0;
    prm.tiles_n = pl.tiles_n;
    prm.timeout_ns = kDefaultTimeoutNs;
    prm.status = st->status_word;
    prm.sk = pl.sk;
    prm.sk_dp_tiles = pl.sk_dp_tiles;
    prm.sk_units = (static_cast<long long>(pl.tiles_n) * ceil_div(M, kBM) - pl.sk_dp_tiles) * pl.num_k_tiles;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    prm.sk_seq = kSkSeqCaptured;
    if (pl.sk) {
        // Partial tiles are written before they are read.  The ready flags
        // keep earlier calls' numbers; this call waits for a new one (see
        // sk_lease), except in a graph capture, where a memset node zeroes
        // them ahead of each replay and the reserved number is used.
        prm.ws = st->noalloc_scratch;
        prm.flags = reinterpret_cast<unsigned int*>(st->noalloc_scratch + kNoAllocMaxCtas * kNoAllocTileFloats);
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(cs, &cap) != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        bool zero = cap != cudaStreamCaptureStatusNone;
        if (!zero) {
            std::lock_guard<std::mutex> lock(st->sk_mu);
            if (st->noalloc_seq + 1 == kSkSeqCaptured) {
                st->noalloc_seq = 0;
                zero = true;
            }
            prm.sk_seq = ++st->noalloc_seq;
        }
        if (zero && cudaMemsetAsync(prm.flags, 0, kNoAllocMaxCtas * sizeof(unsigned int), cs) != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.launch[0].tiles), 1, 1);
    cfg.blockDim = dim3(k.threads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(k.smem_bytes);
    cfg.stream = cs;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;  // finishing CTAs wait on later CTAs
    attr.val.cooperative = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pl.sk ? 1 : 0;
    void* args[3] = {&tmA, &tmB, &prm};
    if (cudaLaunchKernelExC(&cfg, k.fn, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

int run_3xtf32(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
               void* stream, const sgemm_options* opt) {
    int rc = validate(M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (opt && opt->debug_skip_stage < 0) return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    int dev = 0;
    DeviceState* st = nullptr;
    rc = current_device(&dev, &st);
    if (rc != SGEMM_OK) return rc;
    // The tensor-core kernel is fed by tensor maps.  Operands the TMA cannot
    // read (unaligned bases or row strides) are repacked into pitched rows
    // when the product is large enough for that to pay (the same rule as
    // sgemm_f32); otherwise they, and K == 0, take the FFMA kernel, which
    // meets the same contract.
    // Variant: 1 = split-tile kernel (all four TF32 parts in shared memory),
    // 2 = direct-A kernel (A's big part is the TMA tile itself), 3 = the
    // split-tile kernel on 128 x 256 tiles with K-slices of 16, 4 = variant
    // 3 with B's TF32 parts split and transposed in HBM by a pass before the
    // kernel (one read of B and two writes of its size), which leaves the
    // kernel's split warps A only.  Automatic: 4 when the 128 x 256 tiles
    // number at least half the SMs and M >= 1024 (the pass costs ~6/M bytes
    // per flop), 3 when they do with fewer rows, else 1.  Measured on GB300,
    // TFLOP/s for 1 / 3 / 4: 2048^3 155 / 181 / 203, 4096^3 195 / 218 / 261,
    // 8192^3 204 / 243 / 289, 4096 x 4096 x 256 102 / 112 / 116; with fewer
    // tiles 1024^3 61 / 40 / 45, 8192 x 128 x 8192 82 / 51 / 71, 128 x 8192 x
    // 16384 86 / 53 / 22.
    int variant = (opt && opt->math) ? opt->math : 0;
    if (variant == 0)
        variant = 2 * ceil_div(M, kTcBM) * ceil_div(N, 256) < st->sm_count ? 1 : M >= 1024 ? 4 : 3;
    if (variant < 1 || variant > 4) return SGEMM_ERR_INVALID_ARG;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int misaligned = (tma_ok(A, lda) ? 0 : 1) | (tma_ok(B, ldb) ? 0 : 2);
    Repacked packed;
    if (K > 0 && misaligned &&
        2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) >= kRepackMinFlops)
        (void)packed.make(dev, *st, misaligned, M, N, K, A, lda, B, ldb, cs);  // (on failure: the FFMA kernel)
    if (K == 0 || !tma_ok(A, lda) || !tma_ok(B, ldb)) {
        packed.release();
        return run_ffma(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr);
    }
    // Launches: (kernel, tile width, K-slice, grid, first tile, K split).
    // Variants 3 and 4 run whole waves of 128 x 256 tiles; the tiles of a
    // last partial wave run in a second launch of the same kernel with their K
    // slices split between two CTAs each (twice the CTAs at half the work: a
    // fuller wave), the second halves' partial tiles then added into C by
    // add_tiles (a fixed order: deterministic).  4096^3: 3 waves of 152 wide
    // tiles, then 112 CTAs on the last 56 (262 -> 277 TFLOP/s).  Only for
    // K >= 1024: with shorter K the halves' pipeline fill and the pass adding
    // them cost more than the fuller wave gains (4096 x 4096 x 256: 117 ->
    // 105), and the tiles run as one launch.
    struct TcLaunch {
        KernelEntry k;
        int bn, bk;
        long long grid;
        int tile_base, k_split;
        bool pb;  // B's TF32 parts pre-split in HBM (variant 4)
    };
    TcLaunch launches[2];
    int nl = 1;
    const long long tiles_m = ceil_div(M, kTcBM);
    long long split_tiles = 0;  // tiles of the K-split launch
    if (variant >= 3) {
        const KernelEntry wk = variant == 4 ? tf32x3_wide_pb_kernel() : tf32x3_wide_kernel();
        const bool pb = variant == 4;
        const long long wide = tiles_m * ceil_div(N, 256);
        const long long full = (wide / st->sm_count) * st->sm_count;
        if (full > 0 && full < wide && K >= 1024) {
            split_tiles = wide - full;
            launches[0] = {wk, 256, 16, full, 0, 0, pb};
            launches[1] = {wk, 256, 16, 2 * split_tiles, static_cast<int>(full), 2, pb};
            nl = 2;
        } else {
            launches[0] = {wk, 256, 16, wide, 0, 0, pb};
        }
    } else {
        const KernelEntry k = variant == 1 ? tf32x3_kernel() : tf32x3_direct_kernel();
        launches[0] = {k, kTcBN, kTcBK, tiles_m * ceil_div(N, kTcBN), 0, 0, false};
    }
    // The second halves' partial tiles (128 x 256 floats each), from the pool.
    void* ws_split = nullptr;
    if (split_tiles > 0) {
        cudaMemPool_t pool = workspace_pool(dev, *st);
        if (!pool || cudaMallocFromPoolAsync(&ws_split, static_cast<size_t>(split_tiles) * kTcBM * 256 * sizeof(float),
                                             pool, cs) != cudaSuccess) {
            (void)cudaGetLastError();
            packed.release();
            return SGEMM_ERR_CUDA;
        }
    }

    // Variant 4: B's TF32 parts, transposed (N x K4), in a pool buffer.
    void* ws = nullptr;
    float *bt_big = nullptr, *bt_small = nullptr;
    const long long K4 = (static_cast<long long>(K) + 3) / 4 * 4;
    const size_t part = (static_cast<size_t>(N) * K4 * sizeof(float) + 255) & ~size_t{255};
    if (launches[0].pb) {
        cudaMemPool_t pool = workspace_pool(dev, *st);
        if (!pool || cudaMallocFromPoolAsync(&ws, 2 * part, pool, cs) != cudaSuccess) {
            // No room for B's parts (2 N K floats): variant 3's kernels, which
            // split B in shared memory, on the same tiles.
            (void)cudaGetLastError();
            ws = nullptr;
            for (int l = 0; l < nl; ++l) {
                launches[l].k = tf32x3_wide_kernel();
                launches[l].pb = false;
            }
        }
    }
    if (launches[0].pb) {
        bt_big = static_cast<float*>(ws);
        bt_small = reinterpret_cast<float*>(static_cast<char*>(ws) + part);
        rc = split_transpose_b(B, ldb, K, N, bt_big, bt_small, K4, cs);
        if (rc != SGEMM_OK) {
            (void)cudaFreeAsync(ws, cs);
            if (ws_split) (void)cudaFreeAsync(ws_split, cs);
            packed.release();
            return rc;
        }
    }

    rc = SGEMM_OK;
    for (int l = 0; l < nl && rc == SGEMM_OK; ++l) {
        const TcLaunch& ln = launches[l];
        alignas(64) CUtensorMap tmA;
        alignas(64) CUtensorMap tmB;
        alignas(64) CUtensorMap tmB2;
        const CUtensorMapSwizzle swz = ln.bk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        rc = encode_2d(&tmA, A, K, M, lda, ln.bk, kTcBM, swz);
        if (ln.pb) {  // {k, n} boxes of the transposed parts, swizzled like A
            if (rc == SGEMM_OK) rc = encode_2d(&tmB, bt_big, K, N, K4, ln.bk, ln.bn, swz);
            if (rc == SGEMM_OK) rc = encode_2d(&tmB2, bt_small, K, N, K4, ln.bk, ln.bn, swz);
        } else {
            if (rc == SGEMM_OK) rc = encode_2d(&tmB, B, N, K, ldb, ln.bn, ln.bk, CU_TENSOR_MAP_SWIZZLE_NONE);
            tmB2 = tmB;  // (unused)
        }
        if (rc != SGEMM_OK) break;

        TcParams prm;
        prm.M = M;
        prm.N = N;
        prm.K = K;
        prm.C = C;
        prm.ldc = ldc;
        prm.num_k_tiles = static_cast<int>(ceil_div(K, ln.bk));
        prm.tiles_n = static_cast<int>(ceil_div(N, ln.bn));
        prm.tile_base = ln.tile_base;
        prm.k_split = ln.k_split;
        prm.ws = ln.k_split == 2 ? static_cast<float*>(ws_split) : nullptr;
        prm.vec_store = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0) ? 1 : 0;
        prm.skip_stage = opt ? opt->debug_skip_stage : 0;
        prm.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
        prm.status = st->status_word;

        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ln.grid), 1, 1);
        cfg.blockDim = dim3(ln.k.threads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(ln.k.smem_bytes);
        cfg.stream = static_cast<cudaStream_t>(stream);
        cfg.numAttrs = 0;
        void* args4[4] = {&tmA, &tmB, &tmB2, &prm};
        void* args3[3] = {&tmA, &tmB, &prm};  // (the direct-A kernel takes no second B map)
        if (cudaLaunchKernelExC(&cfg, ln.k.fn, variant == 2 ? args3 : args4) != cudaSuccess) {
            (void)cudaGetLastError();
            rc = SGEMM_ERR_CUDA;
        }
    }
    if (rc == SGEMM_OK && split_tiles > 0)
        rc = add_tiles(C, ldc, M, N, static_cast<float*>(ws_split), kTcBM, 256, launches[1].tile_base,
                       static_cast<int>(ceil_div(N, 256)), static_cast<int>(split_tiles), cs);
    if (ws_split) (void)cudaFreeAsync(ws_split, cs);
    if (ws) (void)cudaFreeAsync(ws, cs);
    packed.release();
    return rc;
}

// General form C = alpha * op(A) op(B) + beta * C (see sgemm_f32_gemm).
int run_gemm(int transa, int transb, int M, int N, int K, float alpha, const float* A, int lda, const float* B,
             int ldb, float beta, float* C, int ldc, void* stream) {
    if (transa < 0 || transa > 1 || transb < 0 || transb > 1) return SGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (lda < (transa ? M : K) || ldb < (transb ? K : N) || ldc < N) return SGEMM_ERR_INVALID_ARG;
    const bool product = K > 0 && alpha != 0.f;  // A and B are read
    if (product && M > 0 && !A) return SGEMM_ERR_INVALID_ARG;
    if (product && N > 0 && !B) return SGEMM_ERR_INVALID_ARG;
    if (M > 0 && N > 0 && !C) return SGEMM_ERR_INVALID_ARG;
    const size_t cb = span_bytes(M, N, ldc);
    if (product && (ranges_overlap(C, cb, A, transa ? span_bytes(K, M, lda) : span_bytes(M, K, lda)) ||
                    ranges_overlap(C, cb, B, transb ? span_bytes(N, K, ldb) : span_bytes(K, N, ldb))))
        return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    int dev = 0;
    DeviceState* st = nullptr;
    int rc = current_device(&dev, &st);
    if (rc != SGEMM_OK) return rc;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // No product term (the empty sum, or alpha = 0: A and B are not read).
    if (!product) return scale_c(C, ldc, M, N, beta, cs);
    Scale sc;
    sc.alpha = alpha;
    sc.beta = beta;
    if (!transa && !transb) return run_ffma(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr, &sc);
    // Transposed A that the tensor maps can read stays where it is: the
    // transposed-A kernels load it in its own storage order.  Otherwise, and
    // for a transposed B, one transposing copy into pitched rows per operand
    // (HBM traffic of one read and one write of it), then the product on the
    // copies.
    const bool a_native = transa && tma_ok(A, lda);
    const int copies = (transa && !a_native ? 1 : 0) | (transb ? 2 : 0);
    Repacked packed;
    if (copies) {
        rc = packed.make(dev, *st, copies, M, N, K, A, lda, B, ldb, cs, transa != 0, transb != 0);
        if (rc != SGEMM_OK) return rc;
    }
    rc = run_ffma(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr, &sc, a_native);
    packed.release();
    return rc;
}

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
    std::call_once(st->copy_once, [&] {
        if (cudaStreamCreateWithFlags(&st->copy_in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&st->copy_out, cudaStreamNonBlocking) != cudaSuccess) {
            (void)cudaGetLastError();
            st->copy_in = st->copy_out = nullptr;
        }
    });
    if (!st->copy_in || !st->copy_out) return SGEMM_ERR_CUDA;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaMemPool_t pool = workspace_pool(dev, *st);
    if (!pool) return SGEMM_ERR_CUDA;

    // Row blocks: whole 128-row tiles, up to 8 blocks of >= 512 rows; one
    // block below 2^32 flop (the copies then run before and after the
    // product).  K chunks of B (multiples of 32): 4 when blocked and K >= 1024.
    constexpr int kMaxBlk = 8, kMaxKc = 4;
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

    cudaEvent_t ev_start = nullptr, ev_in_end = nullptr, ev_out_end = nullptr;
    cudaEvent_t ev_a[kMaxBlk] = {}, ev_b[kMaxKc] = {}, ev_done[kMaxBlk] = {};
    auto make_event = [](cudaEvent_t* e) {
        return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    };
    bool ok = make_event(&ev_start) && make_event(&ev_in_end) && make_event(&ev_out_end);
    for (int i = 0; i < nblk && ok; ++i) ok = make_event(&ev_a[i]) && make_event(&ev_done[i]);
    for (int c = 0; c < nkc && ok; ++c) ok = make_event(&ev_b[c]);
    // The copy streams start after the workspace exists (stream order of cs).
    ok = ok && cudaEventRecord(ev_start, cs) == cudaSuccess &&
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
    for (cudaEvent_t e : {ev_start, ev_in_end, ev_out_end})
        if (e) (void)cudaEventDestroy(e);
    for (int i = 0; i < kMaxBlk; ++i) {
        if (ev_a[i]) (void)cudaEventDestroy(ev_a[i]);
        if (ev_done[i]) (void)cudaEventDestroy(ev_done[i]);
    }
    for (int c = 0; c < kMaxKc; ++c)
        if (ev_b[c]) (void)cudaEventDestroy(ev_b[c]);
    if (rc != SGEMM_OK) return rc;
    return ok ? SGEMM_OK : SGEMM_ERR_CUDA;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

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
