// internal.cuh -- helpers shared by the librepops translation units.
//
// Host side: error bookkeeping, per-device properties, range-overlap checks.
// Device side: thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor),
// cp.async and the global nanosecond timer used to bound every wait.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "repops.h"

namespace repops {

// ---------------------------------------------------------------- host ----

// Records `e` as this host thread's last CUDA error; returns REPOPS_ERR_CUDA.
int set_cuda_error(cudaError_t e);

// REPOPS_OK if the last launch on this thread was accepted, else CUDA error.
inline int check_launch() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? REPOPS_OK : set_cuda_error(e);
}

struct DeviceInfo {
    int device = -1;
    int sms = 0;               // multiProcessorCount
    int max_smem_optin = 0;    // sharedMemPerBlockOptin
    int cc_major = 0, cc_minor = 0;
};

// Properties of the current device, cached per device id.
int current_device_info(DeviceInfo *out);

inline bool ranges_overlap(const void *a, uint64_t abytes, const void *b, uint64_t bbytes) {
    if (abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Sticky device status of the GEMM translation unit (bounded waits): the
// word this host thread's launches use (its bound word, else the shared one).
int gemm_read_and_clear_device_status(cudaStream_t stream, unsigned *value);

// A key of the current CUDA context (the driver's context id): addresses
// looked up in one context (a __device__ variable's, say) are only valid
// while the key stays the same.  0 when there is no current context.
int current_context_key(uint64_t *key);

// The device address of the status word this host thread's launches report
// into (its bound word, else the device's shared one).
int status_word_address(unsigned **out);

// Stream-ordered scratch for the entry points: `bytes` on `stream` from the
// library's own memory pool of the current device (one per device and CUDA
// context; how much freed memory it keeps across synchronisations is the
// caller's setting, none by default).  Freed with cudaFreeAsync like any
// stream-ordered allocation.  Returns the CUDA error of the allocation
// (cudaSuccess, or e.g. out of memory).
cudaError_t scratch_malloc(void **ptr, size_t bytes, cudaStream_t stream);

// Makes `stream` wait for everything queued so far on the helper streams a and
// b (either may be null), so that memory released on `stream` afterwards is
// no longer in use by them -- also when the caller stopped half-way on an
// error.  If an event call fails, the helpers are waited for on the host
// instead.  Returns the first error of those calls (cudaSuccess if none).
cudaError_t join_helper_streams(cudaStream_t stream, cudaStream_t a, cudaStream_t b);

// ------------------------------------------------------- debug bounds ----
// The checked build (compiled with -DREPOPS_DEBUG_BOUNDS into
// librepops_debug.so by build.build(checked=True)): the hot-path kernels
// test every global access against the span of the buffer it belongs to; an
// access outside it is skipped and bit 1 of the status word is set, which
// repops_device_status reports as REPOPS_ERR_BOUNDS.  A stand-in for a memory
// sanitizer that never traps or faults.  In the release build the test is the
// constant `true` and compiles away; the spans are then unused parameters.
struct DbgSpan {
    uintptr_t lo = 0, hi = 0;   // the allowed bytes [lo, hi)
};

inline DbgSpan dbg_span(const void *p, uint64_t bytes) {
    DbgSpan s;
    s.lo = reinterpret_cast<uintptr_t>(p);
    s.hi = s.lo + bytes;
    return s;
}

// Bytes of dynamic shared memory this launch was given.
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t v;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}

#ifdef REPOPS_DEBUG_BOUNDS
__device__ __forceinline__ bool dbg_in(const DbgSpan &s, const void *p, uint32_t n, unsigned *status) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if (a >= s.lo && a <= s.hi && n <= s.hi - a) return true;
    if (status) atomicOr(status, 2u);
    return false;
}
// A kernel whose shared-memory need depends on its arguments tests, on entry,
// that the launch gave it that many bytes; if not, it does nothing and sets
// bit 1 of the status word (the same for every thread: no barrier is split).
__device__ __forceinline__ bool dbg_smem(uint64_t need, unsigned *status) {
    if (need <= dynamic_smem_bytes()) return true;
    if (status && threadIdx.x == 0) atomicOr(status, 2u);
    return false;
}
#define REPOPS_DBG_OK(span, p, n, status) ::repops::dbg_in((span), (p), (n), (status))
#define REPOPS_DBG_SMEM_OK(need, status) ::repops::dbg_smem((need), (status))
#else
#define REPOPS_DBG_OK(span, p, n, status) true
#define REPOPS_DBG_SMEM_OK(need, status) true
#endif

// Limit for every device-side wait, in nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// -------------------------------------------------------------- device ----

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Plain arrival (release semantics for this thread's earlier accesses).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete; gives up after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded_ns(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// Waits for phase `parity` of `bar` to complete; gives up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    return mbar_wait_bounded_ns(bar, parity, kWaitLimitNs);
}

// 2-D tiled TMA load of the box at (c0 = inner, c1 = outer) into smem, with
// completion signalled as transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// 3-D tiled TMA load of the box at (c0 = inner, c1 = outer, c2 = batch).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-byte asynchronous global->shared copy; src_bytes == 0 writes zeros.
__device__ __forceinline__ void cp_async_4(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// 16-byte asynchronous global->shared copy bypassing L1; bytes past
// src_bytes (0..16) are written as zeros.  Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace repops
