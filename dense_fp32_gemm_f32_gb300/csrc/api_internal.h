// Internal interface of the library's host code, shared by the translation
// units behind the C entry points (not part of the installed interface): the
// per-device state, the plan of an FFMA call, and the functions those units
// call in one another.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/sgemm.h"
#include "kernels.h"
#include "sgemm_3xtf32_params.h"
#include "sgemm_ffma.cuh"

namespace gb300 {
namespace detail {

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

// Row blocks and K chunks of the host-buffer entry's pipeline (api_host.cu).
constexpr int kHostMaxBlk = 6, kHostMaxKc = 4;
// Its events: start, copies-in done, copies-out done, then per row block
// "block's product done", then per K chunk "chunk's copies in".
constexpr int kHostEvents = 3 + kHostMaxBlk + kHostMaxKc;

struct DeviceState {
    std::once_flag once;
    int status = SGEMM_ERR_CUDA;  // result of the one-time set-up
    int sm_count = 0;
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
    cudaEvent_t host_ev[kHostEvents] = {};  // host-buffer entry: its events, made with the streams
    std::mutex host_mu;               // host-buffer entry: one call enqueues at a time
    std::mutex sk_mu;                        // guards sk_cache, sk_tick and noalloc_seq
    SkScratch sk_cache[kSkCacheEntries];     // per-stream stream-K scratch (sk_lease)
    unsigned long long sk_tick = 0;
    unsigned int noalloc_seq = 0;            // last sequence number of sgemm_f32_noalloc
};

// cuTensorMapEncodeTiled, looked up once (api_device.cu).
extern PFN_cuTensorMapEncodeTiled_v12000 g_encode;

struct SkLease {
    SkScratch* e = nullptr;
    float* ws = nullptr;
    unsigned int* flags = nullptr;
    unsigned int seq = 0;
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Repacking pays once the product is large next to the copy.  Measured on
// GB300 (both operands misaligned, one copy launch for both): 1023 x 1025 x
// 1027 (2^31 flop) 65 us against 69 us with cp.async, 2047 x 2049 x 2051
// +23 %, 4095 x 4097 x 4099 and 8191 x 8193 x 8195 +30 %.
constexpr double kRepackMinFlops = 1073741824.0;  // 2^30

// Misaligned operands are read in place by the residue-class tensor maps
// below 2MNK = kResMaxFlops and repacked from there on.  Measured on GB300
// (both operands misaligned, TFLOP/s, class maps / repacked / cp.async):
// 700 x 900 x 701 27.7 / 23.9 / 24.0, 1023 x 1025 x 1027 37.3 / 34.9 /
// 32.2, 2047 x 2049 x 2051 58.2 / 57.9 / 45.5, 4095 x 4097 x 4099 64.4 /
// 65.8 / 49.0, 8191 x 8193 x 8195 66.5 / 68.7 / 50.2: the copy's cost
// fades with size while the class maps' extra producer work per slice stays.
constexpr double kResMaxFlops = 34359738368.0;  // 2^35

// Rows of tiles per group of the FFMA kernels' tile order (tile_rc): as many
// as keep the group's A row panels within kGroupABytes, between 4 and 16.
constexpr int kGroupRowsMax = 16, kGroupRowsMin = 4;
constexpr long long kGroupABytes = 32ll << 20;

// Fewest 32-deep K slices per tile for which the FFMA kernels write finished
// tiles by tensor-map stores from the staging tile.  Measured on GB300
// (TFLOP/s, direct stores / tensor-map stores): 4096^3 70.0 / 70.3, 8192^3
// 70.4 / 71.0, 128 x 8192 x 16384 68.3 / 68.6, 2048^3 66.8 / 66.6, 1024^3
// 45.9 / 45.5, 4096 x 4096 x 256 62.0 / 59.0 (a barrier pair and 64 KiB of
// shared-memory stores every 8 slices).
constexpr int kTmaStoreMinSlices = 128;

// Shortest K for which the tensor-core entry splits the tiles of a last
// partial wave of 128 x 256 tiles along K (variants 3 and 4).  Measured on
// GB300 with the partial tiles summed in the kernel (TFLOP/s, variant 3 /
// 4, whole / split): 4096^2 x 256 112 / 117 against 93 / 97, x 512 146 / 168
// against 135 / 152, x 768 165 / 195 against 159 / 184, x 1024 174 / 213
// against 174 / 206, 2048^3 181 / 205 either way, 4096^2 x 2048 193 / 240
// against 203 / 244.
constexpr int kTcTailSplitMinK = 2048;

// The library's stream-ordered pool on device `dev` (api_device.cu).
cudaMemPool_t workspace_pool(int dev, DeviceState& st);

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
        // Rows of the copies start on 128-byte boundaries (widths rounded up
        // to 32 floats): the tensor-core kernels' 64-byte box rows then never
        // straddle two 128-byte lines (measured on GB300, sgemm_3xtf32 on
        // 4095 x 4097 x 4099: 186 -> 203 TFLOP/s, on 8191 x 8193 x 8195: 232
        // -> 265, against rows rounded up to 4 floats; sgemm_f32 unchanged).
        const long long K4 = (static_cast<long long>(K) + 31) / 32 * 32;
        const long long N4 = (static_cast<long long>(N) + 31) / 32 * 32;
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

struct Launch {
    int tile_base = 0;  // first output tile
    int tiles = 0;      // output tiles in this launch (grid x)
    int split = 1;      // CTAs per tile along K (cluster z)
};

struct Plan {
    int producer = kProducerTma;
    int math = kMathFfma2;
    int stages = 4;
    int bn = kBN;     // output tile width (kBN or kBNWide)
    int tiles_n = 0;  // tiles per row of tiles
    int tiles_m = 0;  // rows of tiles
    int group_m = 1;  // tile order: rows of tiles per group (tile_rc)
    int a_evict_last = 0;  // A's slices loaded with the L2 evict-last policy
    int b_evict_first = 0; // B's slices loaded with the L2 evict-first policy
    int c_evict_first = 0; // C's tensor-map stores with the L2 evict-first policy
    int num_k_tiles = 0;
    int nlaunch = 1;
    Launch launch[2];
    int sk = 0;           // stream-K: launch[0].tiles CTAs, one per SM
    int sk_dp_tiles = 0;  // tiles taken whole (data-parallel waves) before the stream-K region
    int repack = 0;       // operands copied to 16-byte pitched rows first: bit 0 = A, bit 1 = B
    bool a_mn = false;    // A stored transposed (K x M): the transposed-A kernels
    bool b_nk = false;    // B stored transposed (N x K): the kernels with a B-transposing warp
    int bk = kBK;         // K slice depth (32, or 16 for sgemm_options.tile_k = 16)
    bool res = false;     // A and B read through residue-class tensor maps (any alignment; res_maps.cuh)
    int ec = 0;           // thin column edge: the last N - 128 tiles_n columns, computed with the
                          // last column of tiles (FfmaParams ec; stream-K only)
};

// Epilogue scaling of the general entry: C = alpha * A B + beta * C.
struct Scale {
    float alpha = 1.f, beta = 0.f;
};

// ---- api_device.cu: device set-up, per-stream stream-K scratch
int current_device(int* dev_out, DeviceState** st_out);
int sk_lease(DeviceState& st, cudaStream_t cs, size_t ws_bytes, size_t nflags, SkLease* out);
void sk_return(DeviceState& st, cudaStream_t cs, SkLease& lease);

// ---- api_plan.cu: argument checks and the choice of variant
bool ranges_overlap(const void* a, size_t abytes, const void* b, size_t bbytes);
size_t span_bytes(long long rows, long long cols, long long ld);
int validate(int M, int N, int K, const float* A, int lda, const float* B, int ldb, const float* C, int ldc,
             bool a_mn = false, bool b_nk = false);
bool options_force_variant(const sgemm_options* opt);
int choose_a_layout(int K, const sgemm_options* opt);
bool is_tma(int producer);
KernelEntry ffma_kernel(const Plan& pl);
bool tma_ok(const float* p, int ld);
int make_plan(const DeviceState& st, int M, int N, int K, const float* A, int lda, const float* B, int ldb,
              const sgemm_options* opt, Plan* out, bool a_mn = false, bool b_nk = false, bool scaled = false);
int encode_2d(CUtensorMap* map, const float* base, long long inner, long long outer, long long ld, int box_inner,
              int box_outer, CUtensorMapSwizzle swz);
int encode_res(ResMaps* maps, int* shifts, const float* base, long long rows, long long cols, long long ld,
               int box_inner, int box_outer);
const char* describe_plan(const Plan& pl);
bool small_problem(const DeviceState& st, int M, int N, int K);
bool small_forced_ok(const sgemm_options* opt);

// ---- api_ffma.cu, api_tf32.cu, api_host.cu: the entries' work
int run_ffma(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc, void* stream,
             const sgemm_options* opt, const Scale* scale = nullptr, bool a_mn = false, bool b_nk = false);
int run_ffma_noalloc(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                     void* stream);
int run_gemm(int transa, int transb, int M, int N, int K, float alpha, const float* A, int lda, const float* B,
             int ldb, float beta, float* C, int ldc, void* stream);
int run_3xtf32(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
               void* stream, const sgemm_options* opt);
int run_host(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
             void* stream);

}  // namespace detail
}  // namespace gb300
