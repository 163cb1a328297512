// Per-device set-up (kernel attributes, occupancy figures, the workspace pool,
// the tensor-map encoder), the per-stream stream-K scratch, and the binding of
// a calling thread to its device.
#include "api_internal.h"

namespace gb300 {

// Sticky per-device status word; kernels OR error bits into it.
__device__ unsigned int g_sgemm_status = 0;

namespace detail {

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
            if (set_smem_attr(ffma_kernel_tma_x16(s, math)) != SGEMM_OK) return SGEMM_ERR_CUDA;
            if (set_smem_attr(ffma_kernel_ldg(s, math)) != SGEMM_OK) return SGEMM_ERR_CUDA;
            for (bool scaled : {false, true})
                for (bool edge : {false, true})
                    if (set_smem_attr(ffma_kernel_res(s, math, scaled, edge)) != SGEMM_OK ||
                        set_smem_attr(ffma_kernel_tma_x(s, math, scaled, edge)) != SGEMM_OK)
                        return SGEMM_ERR_CUDA;
            for (bool scaled : {false, true}) {
                if (set_smem_attr(ffma_kernel_bnk(s == 1, scaled)) != SGEMM_OK) return SGEMM_ERR_CUDA;
                if (set_smem_attr(ffma_kernel_amn(s, math, scaled)) != SGEMM_OK) return SGEMM_ERR_CUDA;
            }
        }
    }
    if (set_smem_attr(tf32x3_kernel()) != SGEMM_OK || set_smem_attr(tf32x3_direct_kernel()) != SGEMM_OK ||
        set_smem_attr(tf32x3_wide_kernel()) != SGEMM_OK || set_smem_attr(tf32x3_wide_pb_kernel()) != SGEMM_OK ||
        set_smem_attr(tf32x3_res_kernel()) != SGEMM_OK)
        return SGEMM_ERR_CUDA;
    const KernelEntry ref = ffma_kernel_tma(4, kMathFfma2);
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

}  // namespace detail
}  // namespace gb300
