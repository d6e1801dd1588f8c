// mean_sgd.cu -- fixed-order contributor mean fused with the SGD update.
//
// "Zoo Per-LLM Chain Soundness" §2 Definition "Aggregation rule" (the average
// over the contributor set), §5 "Ordering subroutine" (contributors sorted by
// DID bytes, left fold g(c1) + g(c2) + ... + g(ck), scaled by 1/k),
// "Determinism of left-fold" (round-to-nearest-even, no FMA) and "Update step"
// (theta_t = theta_{t-1} - eta * gbar_t).  Per element e:
//     S = g[o0][e]; S = fl(S + g[o_r][e]) for r = 1..k-1
//     gbar = fl(S / k)
//     theta[e] = fl(theta[e] - fl(eta * gbar))
// The fold order is per element and fixed; elements are independent, so the
// kernel is a coalesced stream: each thread takes float4 chunks, issues all
// gradient loads of a chunk before folding them in order, and writes theta
// back in place.  HBM-bound: (k + 2) * 4 bytes of traffic per element.
//
// Gradients may be stored as binary16 or bfloat16 (widened exactly to binary32
// before the fold; theta stays binary32): (k/2 + 2) * 4 bytes per element.
//
// Division: when k is a power of two, S / k and S * (1/k) are the same real
// number and 1/k is exact in binary32, so both round to the same binary32
// value; the kernel then multiplies.  Otherwise it calls __fdiv_rn, the
// correctly rounded IEEE division.
#include <algorithm>
#include <vector>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"

namespace repops {
namespace {

struct GradPtrs {
    const void *g[REPOPS_MEAN_MAX_CONTRIBUTORS];   // already in fold order
};

// Storage types of the gradients (REPOPS_TYPE_*); widening is exact.
template <int TY>
__device__ __forceinline__ float widen(unsigned short b) {
    if constexpr (TY == REPOPS_TYPE_F16) return __half2float(__ushort_as_half(b));
    else return __uint_as_float(unsigned(b) << 16);
}

template <int TY>
__device__ __forceinline__ float ld1(const void *p, int64_t e) {
    if constexpr (TY == REPOPS_TYPE_F32) return static_cast<const float *>(p)[e];
    else return widen<TY>(static_cast<const unsigned short *>(p)[e]);
}

struct MeanScalars {
    int nC;
    int pow2;        // k is a power of two: multiply by inv
    float count;     // (float)k, exact for k < 2^24
    float inv;       // 1/k when pow2
    float eta;
    // checked build: theta's span, the bytes of one gradient (every gradient
    // access is tested as an offset into [0, gbytes)), the status word
    DbgSpan th, goff;
    unsigned *status;
};

__device__ __forceinline__ float mean_of(float S, const MeanScalars &s) {
    return s.pow2 ? __fmul_rn(S, s.inv) : __fdiv_rn(S, s.count);
}

__device__ __forceinline__ float sgd(float th, float gbar, float eta) {
    return __fsub_rn(th, __fmul_rn(eta, gbar));
}

__device__ __forceinline__ void fold4(float4 &S, const float4 v) {
    S.x = __fadd_rn(S.x, v.x);
    S.y = __fadd_rn(S.y, v.y);
    S.z = __fadd_rn(S.z, v.z);
    S.w = __fadd_rn(S.w, v.w);
}

// Elements 4i .. 4i+3 (16-byte loads for binary32, 8-byte for the half types).
template <int TY>
__device__ __forceinline__ float4 ld4(const void *p, int64_t i) {
    if constexpr (TY == REPOPS_TYPE_F32) {
        return __ldcs(reinterpret_cast<const float4 *>(p) + i);
    } else {
        const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(p) + i);
        return make_float4(widen<TY>(w.x & 0xffffu), widen<TY>(w.x >> 16), widen<TY>(w.y & 0xffffu),
                           widen<TY>(w.y >> 16));
    }
}

// NC > 0: exactly NC contributors, fully unrolled (all loads of a chunk in
// flight together).  NC == 0: any count, loads issued in batches of 8.
template <int TY, int NC>
__global__ void __launch_bounds__(256)
mean_sgd_vec4(const __grid_constant__ GradPtrs gp, const MeanScalars sc, int64_t n4,
              float *__restrict__ theta) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    constexpr uint32_t GB = TY == REPOPS_TYPE_F32 ? 16u : 8u;   // bytes of 4 gradient elements
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += stride) {
        if (!REPOPS_DBG_OK(sc.th, reinterpret_cast<const float4 *>(theta) + i, 16, sc.status) ||
            !REPOPS_DBG_OK(sc.goff, reinterpret_cast<const void *>(uintptr_t(i) * GB), GB, sc.status))
            continue;
        float4 th = __ldcs(reinterpret_cast<const float4 *>(theta) + i);
        float4 S;
        if constexpr (NC > 0) {
            float4 v[NC];
#pragma unroll
            for (int r = 0; r < NC; ++r) v[r] = ld4<TY>(gp.g[r], i);
            S = v[0];
#pragma unroll
            for (int r = 1; r < NC; ++r) fold4(S, v[r]);
        } else {
            constexpr int BATCH = 8;
            S = ld4<TY>(gp.g[0], i);
            int r = 1;
            for (; r + BATCH <= sc.nC; r += BATCH) {
                float4 v[BATCH];
#pragma unroll
                for (int j = 0; j < BATCH; ++j) v[j] = ld4<TY>(gp.g[r + j], i);
#pragma unroll
                for (int j = 0; j < BATCH; ++j) fold4(S, v[j]);
            }
            for (; r < sc.nC; ++r) fold4(S, ld4<TY>(gp.g[r], i));
        }
        th.x = sgd(th.x, mean_of(S.x, sc), sc.eta);
        th.y = sgd(th.y, mean_of(S.y, sc), sc.eta);
        th.z = sgd(th.z, mean_of(S.z, sc), sc.eta);
        th.w = sgd(th.w, mean_of(S.w, sc), sc.eta);
        __stcs(reinterpret_cast<float4 *>(theta) + i, th);
    }
}

// Elements [first, len) one at a time: unaligned buffers, and the len % 4 tail.
template <int TY>
__global__ void __launch_bounds__(256)
mean_sgd_scalar(const __grid_constant__ GradPtrs gp, const MeanScalars sc, int64_t first, int64_t len,
                float *__restrict__ theta) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    constexpr uint32_t GB = TY == REPOPS_TYPE_F32 ? 4u : 2u;   // bytes of one gradient element
    for (int64_t e = first + blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < len; e += stride) {
        if (!REPOPS_DBG_OK(sc.th, theta + e, 4, sc.status) ||
            !REPOPS_DBG_OK(sc.goff, reinterpret_cast<const void *>(uintptr_t(e) * GB), GB, sc.status))
            continue;
        float S = ld1<TY>(gp.g[0], e);
        for (int r = 1; r < sc.nC; ++r) S = __fadd_rn(S, ld1<TY>(gp.g[r], e));
        theta[e] = sgd(theta[e], mean_of(S, sc), sc.eta);
    }
}

template <int TY, int NC>
int launch_vec(const GradPtrs &gp, const MeanScalars &sc, int64_t n4, float *theta, int blocks,
               cudaStream_t s) {
    mean_sgd_vec4<TY, NC><<<blocks, 256, 0, s>>>(gp, sc, n4, theta);
    return check_launch();
}

template <int TY>
int launch_all(const GradPtrs &gp, const MeanScalars &sc, int64_t len, float *theta, bool aligned, int max_blocks,
               cudaStream_t stream) {
    int rc = REPOPS_OK;
    int64_t first_scalar = 0;
    if (aligned) {
        const int64_t n4 = len / 4;
        first_scalar = n4 * 4;
        if (n4 > 0) {
            const int blocks = int(std::min<int64_t>((n4 + 255) / 256, max_blocks));
            switch (sc.nC) {
                case 1: rc = launch_vec<TY, 1>(gp, sc, n4, theta, blocks, stream); break;
                case 2: rc = launch_vec<TY, 2>(gp, sc, n4, theta, blocks, stream); break;
                case 4: rc = launch_vec<TY, 4>(gp, sc, n4, theta, blocks, stream); break;
                case 8: rc = launch_vec<TY, 8>(gp, sc, n4, theta, blocks, stream); break;
                case 16: rc = launch_vec<TY, 16>(gp, sc, n4, theta, blocks, stream); break;
                default: rc = launch_vec<TY, 0>(gp, sc, n4, theta, blocks, stream); break;
            }
            if (rc != REPOPS_OK) return rc;
        }
    }
    if (first_scalar < len) {
        const int64_t n = len - first_scalar;
        const int blocks = int(std::min<int64_t>((n + 255) / 256, max_blocks));
        mean_sgd_scalar<TY><<<blocks, 256, 0, stream>>>(gp, sc, first_scalar, len, theta);
        rc = check_launch();
    }
    return rc;
}

int mean_sgd_typed(int nC, int64_t len, const void *const *ptrs, int gtype, const int *order, float eta,
                   float *theta, cudaStream_t stream) {
    if (gtype != REPOPS_TYPE_F32 && gtype != REPOPS_TYPE_F16 && gtype != REPOPS_TYPE_BF16)
        return REPOPS_ERR_INVALID_ARG;
    if (nC < 1 || nC > REPOPS_MEAN_MAX_CONTRIBUTORS || len < 0) return REPOPS_ERR_INVALID_ARG;
    if (!ptrs || !order) return REPOPS_ERR_INVALID_ARG;
    std::vector<char> seen(size_t(nC), 0);
    for (int r = 0; r < nC; ++r) {
        if (order[r] < 0 || order[r] >= nC || seen[size_t(order[r])]) return REPOPS_ERR_ORDER;
        seen[size_t(order[r])] = 1;
    }
    if (len == 0) return REPOPS_OK;
    if (!theta || len > INT64_MAX / 4) return REPOPS_ERR_INVALID_ARG;
    const uint64_t bytes = uint64_t(len) * 4u;
    const unsigned gsize = gtype == REPOPS_TYPE_F32 ? 4u : 2u;
    const uint64_t gbytes = uint64_t(len) * gsize;
    GradPtrs gp;
    bool aligned = reinterpret_cast<uintptr_t>(theta) % 16 == 0;
    for (int r = 0; r < nC; ++r) {
        const void *g = ptrs[order[r]];
        if (!g) return REPOPS_ERR_INVALID_ARG;
        if (ranges_overlap(theta, bytes, g, gbytes)) return REPOPS_ERR_ALIAS;
        aligned = aligned && reinterpret_cast<uintptr_t>(g) % (4u * gsize) == 0;
        gp.g[r] = g;
    }
    for (int r = nC; r < REPOPS_MEAN_MAX_CONTRIBUTORS; ++r) gp.g[r] = nullptr;

    MeanScalars sc;
    sc.nC = nC;
    sc.pow2 = (nC & (nC - 1)) == 0;
    sc.count = float(nC);
    sc.inv = sc.pow2 ? 1.0f / float(nC) : 0.0f;   // exact: a power of two
    sc.eta = eta;
    sc.th = dbg_span(theta, bytes);
    sc.goff = dbg_span(nullptr, gbytes);
    int rs = status_word_address(&sc.status);
    if (rs != REPOPS_OK) return rs;

    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != REPOPS_OK) return rc;
    const int max_blocks = di.sms * 8;   // 8 CTAs of 256 threads per SM
    if (gtype == REPOPS_TYPE_F16) return launch_all<REPOPS_TYPE_F16>(gp, sc, len, theta, aligned, max_blocks, stream);
    if (gtype == REPOPS_TYPE_BF16)
        return launch_all<REPOPS_TYPE_BF16>(gp, sc, len, theta, aligned, max_blocks, stream);
    return launch_all<REPOPS_TYPE_F32>(gp, sc, len, theta, aligned, max_blocks, stream);
}

}  // namespace
}  // namespace repops

using namespace repops;

extern "C" int repops_fixed_order_mean_sgd(int nC, int64_t len, const float *const *ptrs, const int *order,
                                           float eta, float *theta, cudaStream_t stream) {
    return mean_sgd_typed(nC, len, reinterpret_cast<const void *const *>(ptrs), REPOPS_TYPE_F32, order, eta,
                          theta, stream);
}

extern "C" int repops_fixed_order_mean_sgd_typed(int nC, int64_t len, const void *const *ptrs, int grad_type,
                                                 const int *order, float eta, float *theta, cudaStream_t stream) {
    return mean_sgd_typed(nC, len, ptrs, grad_type, order, eta, theta, stream);
}

extern "C" int repops_fixed_order_mean_sgd_host(int nC, int64_t len, const float *const *ptrs, const int *order,
                                                float eta, float *theta, cudaStream_t stream) {
    if (nC < 1 || nC > REPOPS_MEAN_MAX_CONTRIBUTORS || len < 0) return REPOPS_ERR_INVALID_ARG;
    if (!ptrs || !order) return REPOPS_ERR_INVALID_ARG;
    std::vector<char> seen(size_t(nC), 0);
    for (int r = 0; r < nC; ++r) {
        if (order[r] < 0 || order[r] >= nC || seen[size_t(order[r])]) return REPOPS_ERR_ORDER;
        seen[size_t(order[r])] = 1;
    }
    if (len == 0) return REPOPS_OK;
    if (!theta || len > INT64_MAX / 4) return REPOPS_ERR_INVALID_ARG;
    const uint64_t bytes = uint64_t(len) * 4u;
    for (int r = 0; r < nC; ++r) {
        if (!ptrs[r]) return REPOPS_ERR_INVALID_ARG;
        if (ranges_overlap(theta, bytes, ptrs[r], bytes)) return REPOPS_ERR_ALIAS;
    }
    // element chunks, double-buffered on the device: nC gradient slices and a
    // theta slice per buffer, at most about 1 GiB in all
    const int64_t cap = std::max<int64_t>(1 << 16, (int64_t(1) << 30) / (8 * int64_t(nC + 1)));
    const int64_t ch = std::min<int64_t>(len, std::min<int64_t>(int64_t(1) << 22, cap / 4 * 4));
    const size_t slot = size_t(ch) * 4u;
    void *mem = nullptr;
    if (scratch_malloc(&mem, 2 * size_t(nC + 1) * slot, stream) != cudaSuccess) {
        cudaGetLastError();
        return REPOPS_ERR_ALLOC;
    }
    float *dev = static_cast<float *>(mem);
    auto buf = [&](int b, int r) { return dev + (size_t(b) * (nC + 1) + size_t(r)) * size_t(ch); };
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ready = nullptr, got[2] = {nullptr, nullptr}, back[2] = {nullptr, nullptr};
    cudaError_t e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
        e = cudaEventCreateWithFlags(&got[b], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&back[b], cudaEventDisableTiming);
    }
    // the helper streams start once the allocation is ordered on `stream`
    if (e == cudaSuccess) e = cudaEventRecord(ready, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(in, ready, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(out, ready, 0);
    int rc = REPOPS_OK;
    std::vector<const float *> dptr(static_cast<size_t>(nC));
    for (int64_t c = 0, lo = 0; e == cudaSuccess && rc == REPOPS_OK && lo < len; ++c, lo += ch) {
        const int b = int(c & 1);
        const int64_t n = std::min<int64_t>(ch, len - lo);
        // a buffer is refilled once its previous theta slice has gone back
        if (c >= 2 && (e = cudaStreamWaitEvent(in, back[b], 0)) != cudaSuccess) break;
        for (int r = 0; r < nC && e == cudaSuccess; ++r) {
            e = cudaMemcpyAsync(buf(b, r), ptrs[r] + lo, size_t(n) * 4u, cudaMemcpyHostToDevice, in);
            dptr[size_t(r)] = buf(b, r);
        }
        if (e == cudaSuccess) e = cudaMemcpyAsync(buf(b, nC), theta + lo, size_t(n) * 4u, cudaMemcpyHostToDevice, in);
        if (e == cudaSuccess) e = cudaEventRecord(got[b], in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, got[b], 0);
        if (e != cudaSuccess) break;
        // elements are independent: a slice's update is the whole call's
        rc = mean_sgd_typed(nC, n, reinterpret_cast<const void *const *>(dptr.data()), REPOPS_TYPE_F32, order, eta,
                            buf(b, nC), stream);
        if (rc != REPOPS_OK) break;
        if ((e = cudaEventRecord(got[b], stream)) != cudaSuccess || (e = cudaStreamWaitEvent(out, got[b], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(theta + lo, buf(b, nC), size_t(n) * 4u, cudaMemcpyDeviceToHost, out)) != cudaSuccess ||
            (e = cudaEventRecord(back[b], out)) != cudaSuccess)
            break;
    }
    // `stream` resumes after every copy queued on the helper streams (the last
    // copy back, or what an error left queued); then the memory is released
    const cudaError_t j = join_helper_streams(stream, in, out);
    if (e == cudaSuccess) e = j;
    const cudaError_t f = cudaFreeAsync(mem, stream);
    for (cudaEvent_t x : {ready, got[0], got[1], back[0], back[1]})
        if (x) cudaEventDestroy(x);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
    if (rc != REPOPS_OK) return rc;
    if (e != cudaSuccess) return set_cuda_error(e);
    if (f != cudaSuccess) return set_cuda_error(f);
    return REPOPS_OK;
}
