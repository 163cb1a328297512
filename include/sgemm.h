/*
 * sgemm.h -- C ABI of the GB300 (sm_103a) single-precision matrix multiply.
 *
 * Operation.  For row-major float32 matrices A (M x K) and B (K x N), every
 * entry point below overwrites the row-major M x N matrix C with the product
 *
 *     C[i*ldc + j] = sum_{k=0}^{K-1} A[i*lda + k] * B[k*ldb + j],
 *                    0 <= i < M, 0 <= j < N,
 *
 * the definition C_{i,j} = sum_k A_{i,k} B_{k,j} given in "Hardware
 * acceleration: optimising the memory access pattern of CUDA kernels for
 * matrix multiply", section "computational characteristics of matrix
 * multiplication", with that page's row-major indexing (basic kernel listing)
 * generalised to leading dimensions lda >= K, ldb >= N, ldc >= N.  There is no
 * alpha/beta: C is written, never read.  K == 0 writes zeros (the empty sum);
 * M == 0 or N == 0 is a no-op.
 *
 * Accuracy contract.  Summation order and fused multiply-add contraction are
 * the library's choice.  For every entry, |C - exact| <= 5e-5 * sum_k |A_ik||B_kj|;
 * inputs whose every partial sum is an integer below 2^24 in magnitude (for
 * example entries in {-8..8} with K <= 2^18) give the exact result.
 *
 * Memory.  A, B and C are DEVICE pointers owned by the caller (host
 * pointers for sgemm_f32_host).  C must not overlap A or B.  Rows may be
 * padded (ld > row width); padding is never written and never read.
 *
 * Device memory the library takes itself.  The pages' host code allocates
 * every buffer in the caller; this library also takes scratch of its own,
 * where measurement showed that it pays:
 *  - the stream-K scratch (partial tiles and ready flags, 152 x 128 KiB +
 *    flags on a 152-SM GB300), cudaMalloc'ed on a stream's first stream-K
 *    call and kept for that stream (up to 16 streams) until the process
 *    exits; a call recorded into a CUDA graph takes its stream-K workspace
 *    from the pool below instead;
 *  - from a stream-ordered pool the library creates on each device (cached
 *    up to 256 MiB between calls), freed in stream order at the end of each
 *    call: 16-byte pitched copies of misaligned operands (2MNK >= 2^35),
 *    A's transposed copy (sgemm_options.a_layout = 2), transposed copies of
 *    op(B) = B^T and of an op(A) = A^T the tensor maps cannot read
 *    (sgemm_f32_gemm), B's TF32 parts and the K-split partial tiles and
 *    counters (sgemm_3xtf32), and the device copies of A, B and C
 *    (sgemm_f32_host, which also keeps two copy streams and their events per
 *    device).
 * Entry points that may allocate device memory (machine-read by the tests):
 *   ALLOCATING: sgemm_f32 sgemm_f32_ex sgemm_f32_gemm sgemm_3xtf32 sgemm_3xtf32_ex sgemm_f32_host
 *   NON-ALLOCATING: sgemm_f32_noalloc sgemm_check_status sgemm_status_string sgemm_describe
 * The library's first call on a device (any entry point except
 * sgemm_status_string) also does the one-time device set-up: kernel
 * attributes, occupancy figures, the pool's creation (cudaMemPoolCreate,
 * which reserves no memory by itself) and the tensor-map encoder lookup.
 * Make that first call outside any stream capture.
 *
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL selects the legacy
 * default stream).  Every call enqueues work on that stream and returns without
 * synchronising; the caller synchronises.  Per-device state (the set-up above,
 * the per-stream scratch table, the pool) is created once under locks, so
 * concurrent calls from several host threads are safe.
 *
 * Errors.  Each call returns an sgemm_status.  Argument errors are detected on
 * the host before anything is enqueued.  A kernel that gives up on a bounded
 * wait records SGEMM_ERR_TIMEOUT in a per-device status word, which
 * sgemm_check_status() reads (and clears) after synchronising the stream.
 * Nothing throws across this interface.
 */
#ifndef GB300_SGEMM_H
#define GB300_SGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sgemm_status {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = 1,     /* negative size, ld below row width, NULL with
                                      non-empty operand, C overlapping A or B,
                                      size beyond the documented limits, bad option */
    SGEMM_ERR_UNSUPPORTED = 2,     /* current device is not compute capability
                                      10.3 (the library carries sm_103a code
                                      only), or the requested variant cannot
                                      run on it */
    SGEMM_ERR_CUDA = 3,            /* a CUDA runtime/driver call or the launch failed */
    SGEMM_ERR_TIMEOUT = 4,         /* a kernel abandoned a bounded wait (see
                                      sgemm_check_status) */
    SGEMM_ERR_NOT_IMPLEMENTED = 5  /* the requested path is not built */
} sgemm_status;

/* Size limits: M, N, K and the leading dimensions are int (>= 0), and the
 * number of 128 x 128 output tiles must fit in an int.  Larger requests return
 * SGEMM_ERR_INVALID_ARG. */

/*
 * sgemm_f32 -- C = A x B in float32 on the CUDA cores (FFMA).
 *
 * The main entry.  Picks the kernel variant itself: for small products
 * (2MNK <= 2^28 with at most a quarter as many 128 x 128 tiles as SMs) the
 * 32 x 32-tile small-problem kernel; otherwise 128 x 128 tiles, TMA-fed when
 * A, B have 16-byte aligned bases and row strides (with two warps transposing
 * each A slice in shared memory); misaligned operands are read in place
 * through residue-class tensor maps (SGEMM_PRODUCER_TMA_RES; 2MNK < 2^35,
 * M, K >= 4) or first copied into 16-byte pitched rows (larger products);
 * where neither applies, a cp.async-fed variant reads them.  The schedule is stream-K (one CTA per SM, the work
 * after the last full wave dealt out as K slices) when there are at least two
 * (tile, K slice) units per SM, cluster split-K for smaller outputs.
 * (128 x 256 tiles, a copy of A transposed in HBM and a K-split second
 * launch for the last partial wave are available through sgemm_f32_ex;
 * measured on GB300 none pays, so none is chosen automatically.)
 *   M, N, K      problem sizes (>= 0)
 *   A, lda       device pointer to A, row stride in floats (lda >= K)
 *   B, ldb       device pointer to B, row stride in floats (ldb >= N)
 *   C, ldc       device pointer to C, row stride in floats (ldc >= N)
 *   stream       cudaStream_t as void*
 * A, B and C must be 4-byte aligned (arrays of float); any other alignment
 * returns SGEMM_ERR_INVALID_ARG.
 * A call enqueues the product kernel, preceded, when repacking, by one copy
 * kernel (into a buffer from the library's pool).  The stream-K partial tiles
 * and ready flags live in the scratch the library keeps per stream (its
 * flags carry each call's sequence number, so no memset is needed); a call
 * recorded into a CUDA graph takes a pool workspace whose flags a memset
 * node zeroes instead.  The first stream-K call on a stream allocates
 * (cudaMalloc): make it before any stream capture in the global mode, which
 * such an allocation would invalidate.
 */
int sgemm_f32(int M, int N, int K,
              const float* A, int lda,
              const float* B, int ldb,
              float* C, int ldc,
              void* stream);

/*
 * sgemm_f32_noalloc -- sgemm_f32 for callers that cannot allocate device
 * memory while a call is made.  (The pages this library follows have no
 * counterpart of this entry point.)
 *
 * Who needs it: programs that must keep a fixed device-memory footprint or
 * that hand all device memory to their own allocator up front (a framework's
 * caching allocator, a serving process that reserves everything at start),
 * and latency-critical loops in which a pool allocation could block or fail.
 * sgemm_f32 allocates its stream-K scratch on a stream's first call (and
 * repack buffers from a pool); this entry point takes the scratch from a
 * fixed device array compiled into the library instead, and calls no
 * cudaMalloc, cudaFree or other allocating routine.  The array's ready flags
 * carry each call's sequence number (no memset), except in a stream capture,
 * where a cudaMemsetAsync node (which allocates nothing) clears them ahead
 * of each replay.
 *
 * Same operation, arguments, accuracy contract and errors as sgemm_f32.  It
 * runs the small-problem kernel where sgemm_f32 would, else the FFMA kernel
 * with the stream-K schedule (K == 0: the plain grid, which needs no
 * scratch); misaligned operands are read in place through the residue-class
 * tensor maps (cp.async when M or K < 4), never repacked.
 *
 * Limits and rules:
 *  - The array holds the scratch of at most 160 CTAs: 160 x 64 KiB partial
 *    tiles + 160 flags + 160 x 2 KiB thin-edge partial sums (see
 *    sgemm_options.edge) = 10 MiB + 640 bytes + 320 KiB on every GPU that
 *    loads the library, kept until the process exits.  A call uses one CTA per SM, at
 *    most 160 (a GPU with more SMs still gets a correct, slower result); the
 *    scratch a call needs is bounded by that count, not by M, N or K, and a
 *    call that would need more is rejected with SGEMM_ERR_INVALID_ARG.
 *  - All calls on a device share the array, which keeps the last call's
 *    contents: calls that overlap on the GPU (on different streams, or from
 *    different host threads) race on it and give wrong results.  Order them
 *    on one stream or synchronise between them.
 *  - The first call on each device looks up the array's device address (the
 *    name in host code is only a stand-in) with that device current.  When
 *    it is also the process's first call of this library on the device, it
 *    does the library's one-time device set-up as well (see "Device memory
 *    the library takes itself" above: kernel attributes, the pool's
 *    creation, the tensor-map encoder).  Make that first call before any
 *    stream capture; later calls allocate nothing and create nothing.
 */
int sgemm_f32_noalloc(int M, int N, int K,
                      const float* A, int lda,
                      const float* B, int ldb,
                      float* C, int ldc,
                      void* stream);

/*
 * sgemm_f32_host -- sgemm_f32 on HOST buffers: A, B and C are host pointers
 * (page-locked memory, e.g. from cudaHostAlloc, lets the copies run
 * asynchronously and overlap the product; pageable memory works but
 * serialises).  Same operation, layout rules, accuracy contract and errors as
 * sgemm_f32.
 *
 * The call takes device copies of A, B and C from the library's pool and
 * moves them on two library-owned copy streams.  Products of 2^32 flop and
 * more are pipelined: K is cut into up to four growing chunks, each chunk's
 * columns of A and rows of B are copied in while the product of the chunk
 * before runs (C accumulating on the device), and the last chunk's product
 * runs in up to five shrinking blocks of whole 128-row tiles whose rows of C
 * are copied out while the next block computes.  Smaller products run as
 * one block.  It returns once all of that is enqueued: C holds the result
 * after `stream` is synchronised (all copies are ordered before `stream`'s
 * later work).  The host buffers must stay valid and unmodified until then.
 */
int sgemm_f32_host(int M, int N, int K,
                   const float* A, int lda,
                   const float* B, int ldb,
                   float* C, int ldc,
                   void* stream);

/*
 * sgemm_f32_gemm -- the general form
 *
 *     C = alpha * op(A) op(B) + beta * C      (float32, row-major storage)
 *
 * of the standard GEMM interface (the pages define only the plain product;
 * their optimisation-summary page mentions other storage orders in passing).
 *   transa       0: op(A) = A, stored M x K (lda >= K);
 *                1: op(A) = A^T, A stored K x M (lda >= M)
 *   transb       0: op(B) = B, stored K x N (ldb >= N);
 *                1: op(B) = B^T, B stored N x K (ldb >= K)
 *   alpha, beta  scalars; C is not read when beta == 0 (it may hold NaN or
 *                garbage), and A and B are not read when alpha == 0 or K == 0
 *                (C = beta * C then)
 *   C, ldc       M x N, ldc >= N; must not overlap A or B
 * Same kernels and accuracy contract as sgemm_f32, with the bound
 * |alpha| sum_k |op(A)_ik||op(B)_kj| + |beta||C_ij| per element (exact on
 * integer-valued inputs and integer alpha, beta while every value stays below
 * 2^24).  The epilogue computes fma(beta, C, alpha * (op(A) op(B))).  A
 * transposed operand is first copied, transposed, into pitched rows from the
 * library's pool (one extra read and write of that operand).  Errors as
 * sgemm_f32.
 */
int sgemm_f32_gemm(int transa, int transb,
                   int M, int N, int K,
                   float alpha,
                   const float* A, int lda,
                   const float* B, int ldb,
                   float beta,
                   float* C, int ldc,
                   void* stream);

/*
 * sgemm_3xtf32 -- same operation, signature, accuracy contract and error
 * behaviour as sgemm_f32, computed on the tensor cores (tcgen05): each operand
 * is split into a TF32 "big" part, big = tf32(x), and a TF32 "small" part,
 * small = tf32(x - big), and three TF32 products (small*big + big*small +
 * big*big) are accumulated in float32 in tensor memory.  The dropped terms
 * are below 2^-22 |a||b| each.  The kernels read their operands through
 * tensor maps: operands without 16-byte aligned bases and row strides go to
 * the 128 x 128 kernel on residue-class maps (four per operand, one per
 * class of rows mod 4; M, K >= 4) when that kernel is the choice anyway or
 * 2MNK < 2^30, and are copied into pitched rows first otherwise; K = 0, and
 * misaligned calls with M or K < 4, run the sgemm_f32 kernels.  Tiles of
 * 128 x 256 when those number at
 * least half the SMs (with B's TF32 parts split in a pass before the kernel
 * when M >= 1024), else 128 x 128 (see sgemm_3xtf32_ex).
 * Tensor cores are not on the pages' own path; this entry is reported
 * separately from sgemm_f32.
 */
int sgemm_3xtf32(int M, int N, int K,
                 const float* A, int lda,
                 const float* B, int ldb,
                 float* C, int ldc,
                 void* stream);

/* Producer kinds for sgemm_options.producer. */
enum {
    SGEMM_PRODUCER_AUTO = 0,
    SGEMM_PRODUCER_TMA = 1,      /* tensor-map bulk copies (needs 16-byte alignment) */
    SGEMM_PRODUCER_CPASYNC = 2,  /* 4-byte cp.async with zero fill (any alignment) */
    SGEMM_PRODUCER_TMA_WG = 3,   /* tensor-map bulk copies from a producer warpgroup of its own,
                                    registers split between the warpgroups (producer 40,
                                    consumers 232 per thread); SGEMM_ERR_UNSUPPORTED if the
                                    library's build of that kernel does not allow the split */
    SGEMM_PRODUCER_FUSED = 4,    /* no producer warp: 4-warp CTAs on 128 x 64 tiles, two per SM,
                                    thread 0 issuing the tensor-map copies between its own
                                    multiply-adds (implies tile_n = 64; 2..4 stages, default 4;
                                    no split-K clusters) */
    SGEMM_PRODUCER_TMA_X = 5,    /* tensor-map copies, and two producer warps that
                                    transpose each stage's A slice in shared memory for the
                                    consumers to read per k (the transposed-A read without a
                                    copy of A in HBM; 128 x 128 tiles, 2..4 stages) */
    SGEMM_PRODUCER_LDG = 7,      /* no tensor maps: four producer warps read A's and B's
                                    slice rows from global memory as aligned 16-byte vectors
                                    (any alignment of bases and rows), shift them into place
                                    and store A transposed (m innermost) and B as it is;
                                    128 x 128 tiles, 2..4 stages (default 3).  Measured
                                    slower than repacking or cp.async, so only forced */
    SGEMM_PRODUCER_TMA_RES = 8,  /* operands of any alignment (bases and row pitches that
                                    are whole floats) read in place by tensor maps, four per
                                    operand, one per residue class of rows mod 4: the rows of
                                    a class all start at the same offset (0..3 floats) inside
                                    their 16-byte blocks, so a map based at the block boundary
                                    before the class's first row reads them all, a few floats
                                    early; the two A-transposing warps of SGEMM_PRODUCER_TMA_X
                                    skip those floats, and one more producer warp moves each
                                    B row into place in shared memory.  Needs M >= 4 and
                                    K >= 4; 128 x 128 tiles, paired FMA, 2 to 4 stages
                                    (default 2).  The automatic choice for misaligned
                                    operands (repack = 2 forces the copies instead) */
    SGEMM_PRODUCER_SMALL = 6     /* the small-problem kernel: one 8-warp CTA per 32 x 32 tile
                                    of C, K split across its warps in 32-deep chunks and the
                                    partials summed in a fixed order; bounds-checked 4-byte
                                    loads (any alignment), no pipeline and no waits.  Chosen
                                    automatically when 2MNK <= 2^28 and the 128 x 128 tiles
                                    number at most a quarter of the SMs.  Takes no other
                                    forced field (SGEMM_ERR_INVALID_ARG otherwise) */
};

/*
 * Forced-variant options for ablations and tests.  A zero-initialised struct
 * means "choose automatically" for every field.
 */
typedef struct sgemm_options {
    int producer;       /* SGEMM_PRODUCER_* */
    int split_k;        /* 0 = auto, 1 = none, 2..8 = CTAs per cluster along K */
    int multicast;      /* 0 or 1 = off (the only form built); 2 (two CTAs sharing
                           A's slices by cluster multicast) returns
                           SGEMM_ERR_NOT_IMPLEMENTED: that form is not in
                           this library */
    int math;           /* 0 = auto, 1 = scalar FFMA, 2 = paired FFMA (fma.rn.f32x2) */
    int stages;         /* 0 = auto, else 2..6 shared-memory pipeline stages */
    int debug_skip_stage; /* 0 = off; k > 0: the producer of CTA (0,0,0) never
                             issues its k-th K-slice, so the consumers' bounded
                             wait expires (tests the timeout path) */
    uint64_t timeout_ns;  /* 0 = default (2 s); bound on every in-kernel wait */
    int tail_split;       /* 0 or 1 = off; 2..8 = run the tiles of the last
                             partial wave as a second launch split that many
                             ways along K (only when split_k resolves to 1,
                             the grid exceeds one wave and K has at least
                             4 x tail_split slices of 32) */
    int stream_k;         /* 0 = auto, 1 = off, 2 = on: one CTA per SM; all
                             but the last full wave of tiles run whole, the
                             rest is dealt out evenly as (tile, K slice)
                             units; a tile shared by several CTAs is finished
                             by the CTA holding its first K slice from the
                             others' partial tiles.  Needs a workspace of
                             CTAs x (partial tile + 4 bytes, + 2 KiB with a
                             thin column edge, see edge): the scratch
                             the library keeps per stream (cudaMalloc'ed on
                             the stream's first such call), or, in a stream
                             capture, a pool workspace (see "Device memory
                             the library takes itself"). */
    int tile_n;           /* 0 = auto; 64 = 128 x 64 tiles of the fused
                             producer (SGEMM_PRODUCER_FUSED); 128 = 128 x 128
                             output tiles (8 x 8 per thread); 256 = 128 x 256
                             tiles (8 x 16 per thread,
                             TMA producer warpgroup with the register split,
                             2..4 stages; the stream-K workspace is then
                             CTAs x (128 KiB + 4 bytes)) */
    int repack;           /* 0 = auto, 1 = off, 2 = on: an operand whose base
                             or row pitch is not a multiple of 16 bytes is
                             first copied into rows of ceil(width / 32) x 32
                             floats (a pool workspace of M x K32 and/or
                             K x N32 floats) and the product runs on the
                             tensor-map path; auto = on when no producer is
                             forced and 2MNK >= 2^35 (below that the
                             residue-class tensor maps read such operands in
                             place), 1 = off (the residue-class maps at every
                             size), either way the cp.async producer where
                             the maps cannot run (M or K < 4, a forced
                             choice they do not take) */
    int a_layout;         /* 0 = auto (A stays where it is: the automatic
                             producer transposes its slices in shared memory,
                             SGEMM_PRODUCER_TMA_X), 1 = read A as stored,
                             2 = first copy A transposed (m innermost, a pool
                             workspace of K x M4 floats) and run the
                             transposed-A kernel, whose consumers read each
                             k's A values as two 16-byte vectors */
    int group_m;          /* 0 = auto (as many rows of tiles, 4 to 16, as
                             keep the group's A row panels within 32 MiB:
                             16 at K = 4096, 8 at K = 8192); n >= 1: the
                             output tiles are taken in groups of n rows of
                             tiles, column by column inside a group (odd
                             groups from the right), so that the CTAs
                             running at one time share B column panels (n of
                             them per panel) and A row panels in L2; 1 = row
                             by row.  Larger than the rows of tiles: one
                             group. */
    int l2_hint;          /* 0 = auto (= 4), 1 = no cache policy, 2 = A's
                             slices loaded with the L2 evict-last policy (the
                             A row panels of a tile group stay in L2 across
                             its waves), 3 = that and B's slices with the
                             evict-first policy (tensor-map producers on A
                             and B as stored), 4 = C's tensor-map stores
                             with the evict-first policy (the kernels that
                             store finished tiles from a staging tile) */
    int tile_k;           /* 0 = auto (32), 32, or 16: depth of the K slices
                             the pipeline stages hold (16: the transposing
                             producer, SGEMM_PRODUCER_TMA_X, only; A slices
                             of 64-byte rows with the 64-byte swizzle; 2, 3,
                             4 (default) or 6 stages) */
    int edge;             /* 0 = auto, 1 = off.  Thin column edge: when N mod
                             128 is 1 to 4 and the product runs stream-K on
                             the transposing producer (SGEMM_PRODUCER_TMA_X
                             or SGEMM_PRODUCER_TMA_RES, 32-deep slices,
                             paired FMA, the plain epilogue), those last
                             columns are computed
                             by the CTAs working on the last column of full
                             128 x 128 tiles instead of as a column of tiles
                             of their own (the stream-K workspace then also
                             holds 2 KiB of partial sums per CTA) */
} sgemm_options;

/* sgemm_f32 with forced choices.  Same contract; an unsupported combination
 * returns SGEMM_ERR_INVALID_ARG or SGEMM_ERR_UNSUPPORTED before any launch. */
int sgemm_f32_ex(int M, int N, int K,
                 const float* A, int lda,
                 const float* B, int ldb,
                 float* C, int ldc,
                 void* stream, const sgemm_options* opt);

/* sgemm_3xtf32 with forced choices.  Uses the fields debug_skip_stage,
 * timeout_ns and math, which here selects the tensor-core kernel: 0 = auto
 * (when the 128 x 256 tiles number at least half the SMs: 4 if M >= 1024,
 * else 3; otherwise 1),
 * 1 = split-tile kernel (TF32 big and small parts of both operands stored in
 * shared memory), 2 = direct-A kernel (A's big part is the FP32 tile the TMA
 * lands, read by the tensor core at TF32 precision; only A's small part and
 * B's two parts are stored), both on 128 x 128 tiles; 3 = the split-tile
 * kernel on 128 x 256 tiles with K-slices of 16 (each A element serves twice
 * the columns); 4 = variant 3 with B's TF32 parts split and transposed into a
 * pool buffer first (2 x N x K floats; the kernel loads them with the TMA and
 * splits A only).  3 and 4 run whole waves of 128 x 256 tiles; when K >=
 * 2048 the tiles of a last partial wave run in a second launch with their K
 * slices split between two CTAs, the second halves' partial tiles (a pool
 * workspace of 128 KiB per such tile) added into C, in part order, by the
 * tile's CTA that finishes last.  Variant 1 with at most half as many tiles as
 * SMs splits every tile's nk = ceil(K / 32) K slices among s = min(4, SMs /
 * tiles, nk / 2) CTAs in the same way when nk (s - 1) / s >= 7 + 2 (s - 1)
 * (1024^3: s = 2).  split_k: 0 = automatic, 1 = no K split (any
 * variant), 2..4 = every tile's K slices split among that many CTAs (variant
 * 1, forced or automatic, and at least one 32-deep slice per CTA; for variants
 * 3 and 4, 2 = split the last partial wave's tiles along K whatever K;
 * otherwise SGEMM_ERR_INVALID_ARG).  Other fields are ignored. */
int sgemm_3xtf32_ex(int M, int N, int K,
                    const float* A, int lda,
                    const float* B, int ldb,
                    float* C, int ldc,
                    void* stream, const sgemm_options* opt);

/* Synchronises `stream`, then returns and clears the current device's status
 * word: SGEMM_OK, or SGEMM_ERR_TIMEOUT if any kernel since the last check gave
 * up on a bounded wait (its output is then undefined).  SGEMM_ERR_CUDA if the
 * synchronisation itself fails. */
int sgemm_check_status(void* stream);

/* Static, human-readable name of a status code ("unknown status" otherwise). */
const char* sgemm_status_string(int status);

/* Describes the variant sgemm_f32 would launch for these sizes and pointers on
 * the current device, as a thread-local string such as
 * "tmax/ffma2/s1/st2/sk152" (producer / math / split-K / stages), with, in
 * this order when they apply: "/tailS:T" (T tail tiles run as a second
 * launch split S ways), "/skG" (stream-K over G CTAs), "/nBN" (tiles BN
 * wide, when not 128), "/repackA", "/repackB" or "/repackAB" (operands
 * copied into pitched rows first), "/at" (A read transposed), "/bt" (B
 * stored N x K), "/kBK" (BK-deep slices, when not 32), "/res" (residue-class
 * tensor maps) and "/ecE" (E columns of a thin column edge computed with the
 * last column of tiles; see sgemm_options.edge).  The small-problem kernel
 * reads "small/t32/w8"; an empty output "noop"; arguments sgemm_f32 would
 * refuse "invalid"; no usable device "unavailable".  Host-only; it launches
 * nothing, but sets up the current device on first use. */
const char* sgemm_describe(int M, int N, int K,
                           const float* A, int lda,
                           const float* B, int ldb,
                           const float* C, int ldc);

#ifdef __cplusplus
}
#endif

#endif /* GB300_SGEMM_H */
