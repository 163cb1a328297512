// The FFMA entries' work: sgemm_f32 / sgemm_f32_ex (run_ffma, and the
// small-problem kernel's launch), sgemm_f32_noalloc, and the general form
// sgemm_f32_gemm.
#include "api_internal.h"

namespace gb300 {

// Scratch of sgemm_f32_noalloc: room for the stream-K partial tiles, ready
// flags and thin-edge partial sums of up to kNoAllocMaxCtas CTAs (10 MiB +
// 640 bytes + 320 KiB), a file-scope device array so that the entry point
// needs no allocation.  Every GPU that loads the library holds it until the
// process exits; all calls on a device share it.
constexpr int kNoAllocMaxCtas = 160;
constexpr size_t kNoAllocTileFloats = static_cast<size_t>(kBM) * kBN;  // 128 x 128 tiles only
constexpr size_t kNoAllocEdgeFloats = static_cast<size_t>(kConsumerThreads) * 2;  // FfmaParams ws_edge
constexpr size_t kNoAllocFloats =
    kNoAllocMaxCtas * kNoAllocTileFloats + kNoAllocMaxCtas + kNoAllocMaxCtas * kNoAllocEdgeFloats;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocFloats];

namespace detail {

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
             void* stream, const sgemm_options* opt, const Scale* scale, bool a_mn, bool b_nk) {
    int rc = validate(M, N, K, A, lda, B, ldb, C, ldc, a_mn, b_nk);
    if (rc != SGEMM_OK) return rc;
    if (opt && opt->debug_skip_stage < 0) return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;  // nothing to write; no device work
    int dev = 0;
    DeviceState* st = nullptr;
    rc = current_device(&dev, &st);
    if (rc != SGEMM_OK) return rc;

    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (opt && opt->producer == SGEMM_PRODUCER_SMALL) {
        if (!small_forced_ok(opt) || b_nk) return SGEMM_ERR_INVALID_ARG;
        if (ceil_div(M, kSmallTile) > 65535) return SGEMM_ERR_INVALID_ARG;
        return launch_small(M, N, K, A, lda, B, ldb, C, ldc, stream, scale, a_mn);
    }
    if (!b_nk && !options_force_variant(opt) && !(opt && (opt->a_layout || opt->debug_skip_stage)) &&
        small_problem(*st, M, N, K))
        return launch_small(M, N, K, A, lda, B, ldb, C, ldc, stream, scale, a_mn);
    // A copied transposed for the transposed-A kernels (see choose_a_layout).
    Repacked a_t;
    const int layout = (a_mn || b_nk) ? 0 : choose_a_layout(K, opt);
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
    // and stage choices: the transposed-A kernels have one form.)
    const bool scaled = scale && (scale->alpha != 1.f || scale->beta != 0.f);
    Plan pl;
    rc = make_plan(*st, M, N, K, A, lda, B, ldb, opt, &pl, a_mn, b_nk, scaled);
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
            rc = make_plan(*st, M, N, K, A, lda, B, ldb, &o, &pl, a_mn, b_nk, scaled);
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

    const KernelEntry k = pl.res ? ffma_kernel_res(pl.stages, pl.math, scaled, pl.ec > 0)
                          : pl.b_nk ? ffma_kernel_bnk(pl.a_mn, scaled)
                          : pl.a_mn ? (pl.bn == kBN ? ffma_kernel_amn(pl.stages, pl.math, scaled)
                                                  : scaled ? KernelEntry{nullptr, 0, 0} : ffma_kernel(pl))
                          : scaled ? (pl.producer == kProducerTmaX  ? ffma_kernel_tma_x(pl.stages, pl.math, true)
                                      : pl.bn == kBN               ? ffma_kernel_scaled(pl.producer, pl.stages, pl.math)
                                                                   : KernelEntry{nullptr, 0, 0})
                                   : ffma_kernel(pl);
    if (!k.fn) {
        release_pack();
        return SGEMM_ERR_INVALID_ARG;
    }

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    alignas(64) CUtensorMap tmC;
    std::memset(&tmA, 0, sizeof tmA);
    std::memset(&tmB, 0, sizeof tmB);
    std::memset(&tmC, 0, sizeof tmC);
    // Tensor-map stores of C need 16-byte rows and base, and N a multiple of
    // 4: measured on GB300, a store whose box crosses the end of a row also
    // writes the rest of the 16-byte group holding the last column (the row
    // padding of C, which the contract leaves untouched).  They pay only for
    // long K loops (kTmaStoreMinSlices).
    const bool c_aligned = tma_ok(C, ldc) && N % 4 == 0 && pl.num_k_tiles >= kTmaStoreMinSlices;
    if (k.tma_store && c_aligned) {
        rc = encode_2d(&tmC, C, N, M, ldc, kBN, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);  // {n, m} boxes of 128 x 128
        if (rc != SGEMM_OK) {
            release_pack();
            return rc;
        }
    }
    // Residue-class maps (pl.res): four per operand, boxes of 36 k x 32 rows
    // of A and 132 columns x 8 rows of B (res_maps.cuh).
    ResMaps resA, resB;
    std::memset(&resA, 0, sizeof resA);
    std::memset(&resB, 0, sizeof resB);
    int a_shift = 0, b_shift = 0;
    if (pl.res) {
        rc = encode_res(&resA, &a_shift, A, M, K, lda, kResABox, kBM / 4);
        if (rc == SGEMM_OK) rc = encode_res(&resB, &b_shift, B, K, N, ldb, kResBBox, kBK / 4);
        if (rc != SGEMM_OK) {
            release_pack();
            return rc;
        }
    } else if (is_tma(pl.producer)) {
        rc = pl.a_mn ? encode_2d(&tmA, A, M, K, lda, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_NONE)  // {m, k} boxes of 128 x 32
             : pl.bk == kBK16 ? encode_2d(&tmA, A, K, M, lda, kBK16, kBM, CU_TENSOR_MAP_SWIZZLE_64B)
                              : encode_2d(&tmA, A, K, M, lda, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc == SGEMM_OK)
            rc = pl.b_nk ? encode_2d(&tmB, B, K, N, ldb, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B)  // {k, n} boxes of 32 x 128
                         : encode_2d(&tmB, B, N, K, ldb, pl.bn, pl.bk, CU_TENSOR_MAP_SWIZZLE_NONE);
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
    prm.vec_store = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0) ? 1 : 0;
    prm.tiles_n = pl.tiles_n;
    prm.tiles_m = pl.tiles_m;
    prm.group_m = pl.group_m;
    prm.a_evict_last = pl.a_evict_last;
    prm.b_evict_first = pl.b_evict_first;
    prm.c_evict_first = pl.c_evict_first;
    prm.tma_store = (k.tma_store && c_aligned) ? 1 : 0;
    prm.skip_stage = opt ? opt->debug_skip_stage : 0;
    prm.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
    prm.status = st->status_word;
    prm.alpha = scale ? scale->alpha : 1.f;
    prm.beta = scale ? scale->beta : 0.f;
    prm.a_shift = a_shift;
    prm.b_shift = b_shift;
    prm.sk = pl.sk;
    prm.sk_dp_tiles = pl.sk_dp_tiles;
    prm.sk_units = (static_cast<long long>(pl.tiles_n) * ceil_div(M, kBM) - pl.sk_dp_tiles) * pl.num_k_tiles;
    prm.ec = pl.ec;
    prm.ws = nullptr;
    prm.ws_edge = nullptr;
    prm.flags = nullptr;
    prm.sk_seq = kSkSeqCaptured;

    // Stream-K workspace: one partial tile and one flag per CTA (and, with a
    // thin column edge, 256 partial column pairs), from the stream's own
    // scratch (sk_lease) or, while the stream is being captured into a graph,
    // from the library's stream-ordered pool for this call with its flags
    // zeroed by a memset (stream order makes concurrent calls on different
    // streams use different workspaces).
    void* ws = nullptr;
    SkLease lease;
    if (pl.sk) {
        const size_t G = static_cast<size_t>(pl.launch[0].tiles);
        const size_t tile_bytes = static_cast<size_t>(kBM) * pl.bn * sizeof(float);
        const size_t edge_bytes = pl.ec ? G * kConsumerThreads * sizeof(float2) : 0;
        if (sk_lease(*st, cs, G * tile_bytes + edge_bytes, G, &lease) == SGEMM_OK) {
            prm.ws = lease.ws;
            prm.flags = lease.flags;
            prm.sk_seq = lease.seq;
        } else {
            cudaMemPool_t pool = workspace_pool(dev, *st);
            if (!pool || cudaMallocFromPoolAsync(&ws, G * tile_bytes + edge_bytes + G * sizeof(unsigned int), pool,
                                                 cs) != cudaSuccess) {
                (void)cudaGetLastError();
                release_pack();
                return SGEMM_ERR_CUDA;
            }
            prm.ws = static_cast<float*>(ws);
            prm.flags = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + G * tile_bytes + edge_bytes);
            if (cudaMemsetAsync(prm.flags, 0, G * sizeof(unsigned int), cs) != cudaSuccess) {
                (void)cudaGetLastError();
                (void)cudaFreeAsync(ws, cs);
                release_pack();
                return SGEMM_ERR_CUDA;
            }
        }
        if (pl.ec) prm.ws_edge = reinterpret_cast<float2*>(reinterpret_cast<char*>(prm.ws) + G * tile_bytes);
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
            attr.val.clusterDim.x = 1;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = ln.split;
        }
        cfg.attrs = &attr;
        cfg.numAttrs = (pl.sk || ln.split > 1) ? 1 : 0;
        void* args[4] = {pl.res ? static_cast<void*>(&resA) : &tmA, pl.res ? static_cast<void*>(&resB) : &tmB, &tmC,
                         &prm};
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
    o.repack = 1;  // repacking would allocate: misaligned operands take the residue-class maps, else cp.async
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
    alignas(64) CUtensorMap tmC;
    std::memset(&tmA, 0, sizeof tmA);
    std::memset(&tmB, 0, sizeof tmB);
    std::memset(&tmC, 0, sizeof tmC);
    const bool c_tma = k.tma_store && tma_ok(C, ldc) && N % 4 == 0 &&
                       pl.num_k_tiles >= kTmaStoreMinSlices;  // (as in run_ffma)
    if (c_tma) {
        rc = encode_2d(&tmC, C, N, M, ldc, kBN, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != SGEMM_OK) return rc;
    }
    ResMaps resA, resB;
    std::memset(&resA, 0, sizeof resA);
    std::memset(&resB, 0, sizeof resB);
    int a_shift = 0, b_shift = 0;
    if (pl.res) {
        rc = encode_res(&resA, &a_shift, A, M, K, lda, kResABox, kBM / 4);
        if (rc == SGEMM_OK) rc = encode_res(&resB, &b_shift, B, K, N, ldb, kResBBox, kBK / 4);
        if (rc != SGEMM_OK) return rc;
    } else if (is_tma(pl.producer)) {
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
    prm.vec_store = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0) ? 1 : 0;
    prm.tile_base = 0;
    prm.tiles_n = pl.tiles_n;
    prm.tiles_m = pl.tiles_m;
    prm.group_m = pl.group_m;
    prm.a_evict_last = pl.a_evict_last;
    prm.b_evict_first = pl.b_evict_first;
    prm.c_evict_first = pl.c_evict_first;
    prm.tma_store = c_tma ? 1 : 0;
    prm.timeout_ns = kDefaultTimeoutNs;
    prm.status = st->status_word;
    prm.a_shift = a_shift;
    prm.b_shift = b_shift;
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
        prm.ec = pl.ec;
        prm.ws_edge = pl.ec ? reinterpret_cast<float2*>(st->noalloc_scratch + kNoAllocMaxCtas * kNoAllocTileFloats +
                                                          kNoAllocMaxCtas)
                            : nullptr;
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
    void* args[4] = {pl.res ? static_cast<void*>(&resA) : &tmA, pl.res ? static_cast<void*>(&resB) : &tmB, &tmC,
                     &prm};
    if (cudaLaunchKernelExC(&cfg, k.fn, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
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
    // Arrays of float: 4-byte aligned (the copies below index them as such).
    if (((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 3u) != 0)
        return SGEMM_ERR_INVALID_ARG;
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
    // A transposed operand that the tensor maps can read stays where it is:
    // the transposed-A kernels load A in its own storage order, and a B
    // stored N x K is loaded in slices of 128 n x 32 k that a producer warp
    // transposes in shared memory (products too small for the 128 x 128
    // kernels, which go to the small-problem kernel, take the copy below).
    // Otherwise one transposing copy into pitched rows per operand (HBM
    // traffic of one read and one write of it), then the product on the
    // copies.
    const bool a_native = transa && tma_ok(A, lda);
    const bool b_native = transb && tma_ok(B, ldb) && !small_problem(*st, M, N, K);
    const int copies = (transa && !a_native ? 1 : 0) | (transb && !b_native ? 2 : 0);
    Repacked packed;
    if (copies) {
        rc = packed.make(dev, *st, copies, M, N, K, A, lda, B, ldb, cs, transa != 0, transb != 0);
        if (rc != SGEMM_OK) return rc;
    }
    rc = run_ffma(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr, &sc, a_native, b_native);
    packed.release();
    return rc;
}

}  // namespace detail
}  // namespace gb300
