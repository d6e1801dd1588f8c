// abi.cu -- library-wide C-ABI entry points: build manifest, status strings,
// CUDA error bookkeeping, device properties, the contributor sort, the sticky
// device status word and the stream-ordered scratch pool.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.cuh"

#ifndef REPOPS_BUILD_FLAGS
#define REPOPS_BUILD_FLAGS "unknown"
#endif

namespace repops {

namespace {
thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
struct CachedInfo {
    std::atomic<int> ready{0};
    DeviceInfo info;
};
CachedInfo g_info[kMaxDevices];
}  // namespace

int set_cuda_error(cudaError_t e) {
    t_last_cuda_error = int(e);
    return REPOPS_ERR_CUDA;
}

int current_device_info(DeviceInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return REPOPS_ERR_UNSUPPORTED;
    CachedInfo &c = g_info[dev];
    if (!c.ready.load(std::memory_order_acquire)) {
        DeviceInfo d;
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return set_cuda_error(e);
        c.info = d;   // identical values if two threads race here
        c.ready.store(1, std::memory_order_release);
    }
    *out = c.info;
    return REPOPS_OK;
}

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_ctx_once;

template <class Fn>
Fn driver_entry(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<Fn>(p);
    return nullptr;
}
}  // namespace

int current_context_key(uint64_t *key) {
    std::call_once(g_ctx_once, [] {
        g_ctx_get_current = driver_entry<CtxGetCurrentFn>("cuCtxGetCurrent");
        g_ctx_get_id = driver_entry<CtxGetIdFn>("cuCtxGetId");
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return REPOPS_ERR_UNSUPPORTED;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return REPOPS_ERR_UNSUPPORTED;
    if (!ctx) {
        // a host thread whose first runtime call this is: the runtime makes
        // the current device's primary context current
        cudaError_t e = cudaFree(nullptr);
        if (e != cudaSuccess) return set_cuda_error(e);
        if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return REPOPS_ERR_UNSUPPORTED;
    }
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return REPOPS_ERR_UNSUPPORTED;
    *key = uint64_t(id) + 1u;   // never 0
    return REPOPS_OK;
}

namespace {
// The scratch pool of each device, created in the CUDA context current at
// the first allocation and again when that context changes (after
// cudaDeviceReset the old handle is gone with its context).  `keep` is the
// caller's setting (repops_scratch_set_keep_bytes), 0 by default: the pool
// then hands freed memory back at every synchronisation, as the device's
// default pool does, and the library holds no memory between calls.  A call
// made after a synchronisation then maps its scratch again: ~120 us of host
// time with the GPU idle if nothing else was queued (measured on a GB300,
// synchronised after every call: a 1536^3 GEMM 318 us a call, 242 us with
// the scratch kept; 2048^3 598 -> 522 us).
struct ScratchPool {
    std::mutex mu;
    uint64_t ctx_key = 0;
    cudaMemPool_t pool = nullptr;
    uint64_t keep = 0;
};
ScratchPool g_scratch_pool[kMaxDevices];

// The current device's pool (created if needed) and its slot.
int scratch_pool(cudaMemPool_t *pool, ScratchPool **slot = nullptr) {
    *pool = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return REPOPS_ERR_UNSUPPORTED;
    uint64_t key = 0;
    int rc = current_context_key(&key);
    if (rc != REPOPS_OK) return rc;
    ScratchPool &s = g_scratch_pool[dev];
    std::lock_guard<std::mutex> lock(s.mu);
    if (s.ctx_key != key || !s.pool) {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof props);
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if ((e = cudaMemPoolCreate(&p, &props)) != cudaSuccess) return set_cuda_error(e);
        uint64_t keep = s.keep;
        if ((e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return set_cuda_error(e);
        }
        s.pool = p;
        s.ctx_key = key;
    }
    *pool = s.pool;
    if (slot) *slot = &s;
    return REPOPS_OK;
}
}  // namespace

cudaError_t scratch_malloc(void **ptr, size_t bytes, cudaStream_t stream) {
    cudaMemPool_t pool = nullptr;
    if (scratch_pool(&pool) != REPOPS_OK || !pool) {
        // no pool of our own (it could not be created): the device's default one
        cudaGetLastError();
        return cudaMallocAsync(ptr, bytes, stream);
    }
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

cudaError_t join_helper_streams(cudaStream_t stream, cudaStream_t a, cudaStream_t b) {
    cudaError_t first = cudaSuccess;
    for (cudaStream_t h : {a, b}) {
        if (!h) continue;
        cudaEvent_t ev = nullptr;
        cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventRecord(ev, h);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev, 0);
        if (ev) cudaEventDestroy(ev);
        if (e != cudaSuccess) {
            cudaStreamSynchronize(h);
            if (first == cudaSuccess) first = e;
        }
    }
    return first;
}

}  // namespace repops

using namespace repops;

extern "C" const char *repops_version(void) {
    return "librepops 0.1.0; arch sm_103a; fp32 IEEE-754 round-to-nearest-even, no FMA, no FTZ, "
           "no tensor cores; gemm tiles 128x128/256t 8x8, 64x128/128t 8x8, 128x64/128t 8x8, "
           "64x64/128t 8x4, 32x64/128t 4x4, BK 32, loaders TMA(128B swizzle)+cp.async; "
           "mean+sgd left fold, divide by count; merkle sha256 leaf 0x00 node 0x01 promote-odd; "
           "flags: " REPOPS_BUILD_FLAGS;
}

extern "C" const char *repops_status_string(int status) {
    switch (status) {
        case REPOPS_OK: return "ok";
        case REPOPS_ERR_INVALID_ARG: return "invalid argument";
        case REPOPS_ERR_ALIAS: return "output overlaps an input";
        case REPOPS_ERR_ORDER: return "contributor order is not a permutation or identifiers repeat";
        case REPOPS_ERR_CUDA: return "CUDA runtime error";
        case REPOPS_ERR_TIMEOUT: return "a bounded device-side wait gave up";
        case REPOPS_ERR_ALLOC: return "scratch allocation failed";
        case REPOPS_ERR_UNSUPPORTED: return "outside the supported limits";
        case REPOPS_ERR_BOUNDS: return "a checked access fell outside its buffer (checked build)";
        default: return "unknown status";
    }
}

extern "C" int repops_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int repops_device_status(cudaStream_t stream, int *status_out) {
    if (!status_out) return REPOPS_ERR_INVALID_ARG;
    unsigned v = 0;
    int rc = gemm_read_and_clear_device_status(stream, &v);
    if (rc != REPOPS_OK) return rc;
    *status_out = (v & 2u) ? REPOPS_ERR_BOUNDS : v ? REPOPS_ERR_TIMEOUT : REPOPS_OK;
    return REPOPS_OK;
}

extern "C" int repops_scratch_release(void) {
    cudaMemPool_t pool = nullptr;
    int rc = scratch_pool(&pool);
    if (rc != REPOPS_OK) return rc;
    const cudaError_t e = cudaMemPoolTrimTo(pool, 0);
    return e == cudaSuccess ? REPOPS_OK : set_cuda_error(e);
}

extern "C" int repops_scratch_set_keep_bytes(uint64_t bytes) {
    cudaMemPool_t pool = nullptr;
    ScratchPool *slot = nullptr;
    int rc = scratch_pool(&pool, &slot);
    if (rc != REPOPS_OK) return rc;
    std::lock_guard<std::mutex> lock(slot->mu);
    uint64_t v = bytes;
    const cudaError_t e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &v);
    if (e != cudaSuccess) return set_cuda_error(e);
    slot->keep = bytes;
    return REPOPS_OK;
}

extern "C" int repops_scratch_reserved_bytes(uint64_t *bytes_out) {
    if (!bytes_out) return REPOPS_ERR_INVALID_ARG;
    cudaMemPool_t pool = nullptr;
    int rc = scratch_pool(&pool);
    if (rc != REPOPS_OK) return rc;
    cuuint64_t v = 0;
    const cudaError_t e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &v);
    if (e != cudaSuccess) return set_cuda_error(e);
    *bytes_out = uint64_t(v);
    return REPOPS_OK;
}

// "Zoo Per-LLM Chain Soundness" §5 "Ordering subroutine": contributors sorted
// lexicographically by DID bytes (unsigned; a proper prefix first).
extern "C" int repops_sort_ids(int n, const uint8_t *ids, const int64_t *offsets, const int64_t *lengths,
                               int *order_out) {
    if (n < 0) return REPOPS_ERR_INVALID_ARG;
    if (n == 0) return REPOPS_OK;
    if (!ids || !offsets || !lengths || !order_out) return REPOPS_ERR_INVALID_ARG;
    for (int r = 0; r < n; ++r)
        if (offsets[r] < 0 || lengths[r] < 0) return REPOPS_ERR_INVALID_ARG;
    auto less = [&](int a, int b) {
        const int64_t la = lengths[a], lb = lengths[b];
        const int c = std::memcmp(ids + offsets[a], ids + offsets[b], size_t(std::min(la, lb)));
        return c != 0 ? c < 0 : la < lb;
    };
    std::vector<int> idx(static_cast<size_t>(n));
    for (int r = 0; r < n; ++r) idx[size_t(r)] = r;
    std::stable_sort(idx.begin(), idx.end(), less);
    for (int r = 1; r < n; ++r)
        if (!less(idx[size_t(r - 1)], idx[size_t(r)])) return REPOPS_ERR_ORDER;
    std::copy(idx.begin(), idx.end(), order_out);
    return REPOPS_OK;
}
