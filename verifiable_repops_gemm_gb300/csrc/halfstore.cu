// halfstore.cu -- half-precision storage around the binary32 order-fixed path,
// and rolling hashes of uint32 batch rows.
//
// "Verde与RepOps" §3.3 (IEEE-754 hardware needed; FP16 support limited), §5.3
// (lower-precision training as future work).  The pages fix no format rules;
// the library's: binary16 and bfloat16 elements are widened exactly to
// binary32 (every half value is a binary32 value), the binary32 order-fixed
// kernels compute, and a half result is narrowed once with the IEEE
// round-to-nearest-even conversion (cvt.rn).  The conversions here are the
// only place where a half type meets the arithmetic.
//
// ZKDV page, proof.start(rolling_window=...): rolling hashes within each
// committed row of a rectangular uint32 batch.  The page names no hash; the
// library's is Rabin-Karp modulo the Mersenne prime 2^61 - 1.  Each thread
// takes 64 consecutive window starts of one row: Horner's rule for the first,
// then h' = h * B - w_out * B^W + w_in for the rest -- exact modular integers,
// so the split of a row across threads does not change a bit.  With
// B = 2^32 + 15 the products by B are 61-bit rotations (roll61.cuh).
// Windows up to 1024 words stage a warp's words and hashes in shared memory
// (coalesced global accesses); longer ones read global memory directly.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"
#include "roll61.cuh"

namespace repops {
namespace {

bool known_type(int t) { return t == REPOPS_TYPE_F32 || t == REPOPS_TYPE_F16 || t == REPOPS_TYPE_BF16; }
constexpr unsigned type_size(int t) { return t == REPOPS_TYPE_F32 ? 4u : 2u; }

// ------------------------------------------------------------ conversions ----

template <int TY>
__device__ __forceinline__ float load_f32(const void *p, int64_t i) {
    if constexpr (TY == REPOPS_TYPE_F32) return static_cast<const float *>(p)[i];
    else if constexpr (TY == REPOPS_TYPE_F16) return __half2float(static_cast<const __half *>(p)[i]);
    else return __uint_as_float(unsigned(static_cast<const unsigned short *>(p)[i]) << 16);
}

template <int TY>
__device__ __forceinline__ void store_from_f32(void *p, int64_t i, float v) {
    if constexpr (TY == REPOPS_TYPE_F32) static_cast<float *>(p)[i] = v;
    else if constexpr (TY == REPOPS_TYPE_F16) static_cast<__half *>(p)[i] = __float2half_rn(v);
    else static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
}

// Elements 4i .. 4i+3 (16-byte accesses for binary32, 8-byte for the halves).
template <int TY>
__device__ __forceinline__ float4 load4(const void *p, int64_t i) {
    if constexpr (TY == REPOPS_TYPE_F32) {
        return __ldcs(reinterpret_cast<const float4 *>(p) + i);
    } else {
        const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(p) + i);
        const unsigned short h[4] = {(unsigned short)(w.x & 0xffffu), (unsigned short)(w.x >> 16),
                                     (unsigned short)(w.y & 0xffffu), (unsigned short)(w.y >> 16)};
        return make_float4(load_f32<TY>(h, 0), load_f32<TY>(h, 1), load_f32<TY>(h, 2), load_f32<TY>(h, 3));
    }
}

template <int TY>
__device__ __forceinline__ void store4(void *p, int64_t i, float4 v) {
    if constexpr (TY == REPOPS_TYPE_F32) {
        __stcs(reinterpret_cast<float4 *>(p) + i, v);
    } else {
        unsigned short h[4];
        store_from_f32<TY>(h, 0, v.x);
        store_from_f32<TY>(h, 1, v.y);
        store_from_f32<TY>(h, 2, v.z);
        store_from_f32<TY>(h, 3, v.w);
        __stcs(reinterpret_cast<uint2 *>(p) + i, make_uint2(h[0] | (unsigned(h[1]) << 16), h[2] | (unsigned(h[3]) << 16)));
    }
}

// n contiguous elements; vec: both buffers aligned to 4 elements, so whole
// groups of four move with one vector access each.  Each thread converts the
// same elements it reads, so an in-place conversion between types of one size
// is safe.
template <int S, int D>
__global__ void __launch_bounds__(256)
convert_1d_kernel(int64_t n, const void *src, void *dst, int vec) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const int64_t first = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    int64_t done = 0;
    if (vec) {
        const int64_t n4 = n / 4;
        for (int64_t i = first; i < n4; i += stride) store4<D>(dst, i, load4<S>(src, i));
        done = n4 * 4;
    }
    for (int64_t e = done + first; e < n; e += stride) store_from_f32<D>(dst, e, load_f32<S>(src, e));
}

// rows x cols elements: source element (r, c) at src[r*lds + c], destination at
// dst[r*ldd + c]; rows over blockIdx.y, columns over the x dimension.
template <int S, int D>
__global__ void __launch_bounds__(256)
convert_2d_kernel(int64_t rows, int64_t cols, const void *src, int64_t lds, void *dst, int64_t ldd) {
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y)
        for (int64_t c = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; c < cols; c += int64_t(gridDim.x) * blockDim.x)
            store_from_f32<D>(dst, r * ldd + c, load_f32<S>(src, r * lds + c));
}

template <int S, int D>
int launch_convert_pair(int64_t rows, int64_t cols, const void *src, int64_t lds, void *dst, int64_t ldd,
                        cudaStream_t s) {
    DeviceInfo di;
    const int sms = current_device_info(&di) == REPOPS_OK ? di.sms : 152;
    if (rows == 1 || (lds == cols && ldd == cols)) {
        const int64_t n = rows * cols;
        const int vec = reinterpret_cast<uintptr_t>(src) % (4u * type_size(S)) == 0 &&
                        reinterpret_cast<uintptr_t>(dst) % (4u * type_size(D)) == 0;
        const int blocks = int(std::min<int64_t>((n / 4 + 255) / 256 + 1, int64_t(sms) * 16));
        convert_1d_kernel<S, D><<<blocks, 256, 0, s>>>(n, src, dst, vec);
    } else {
        const int gx = int(std::min<int64_t>((cols + 255) / 256, 32));
        const int gy = int(std::min<int64_t>(rows, 65535));
        convert_2d_kernel<S, D><<<dim3(gx, gy), 256, 0, s>>>(rows, cols, src, lds, dst, ldd);
    }
    return check_launch();
}

template <int S>
int launch_convert_to(int dtype, int64_t rows, int64_t cols, const void *src, int64_t lds, void *dst,
                      int64_t ldd, cudaStream_t s) {
    if (dtype == REPOPS_TYPE_F32) return launch_convert_pair<S, REPOPS_TYPE_F32>(rows, cols, src, lds, dst, ldd, s);
    if (dtype == REPOPS_TYPE_F16) return launch_convert_pair<S, REPOPS_TYPE_F16>(rows, cols, src, lds, dst, ldd, s);
    return launch_convert_pair<S, REPOPS_TYPE_BF16>(rows, cols, src, lds, dst, ldd, s);
}

int launch_convert(int stype, int dtype, int64_t rows, int64_t cols, const void *src, int64_t lds, void *dst,
                   int64_t ldd, cudaStream_t s) {
    if (rows == 0 || cols == 0) return REPOPS_OK;
    if (stype == REPOPS_TYPE_F32) return launch_convert_to<REPOPS_TYPE_F32>(dtype, rows, cols, src, lds, dst, ldd, s);
    if (stype == REPOPS_TYPE_F16) return launch_convert_to<REPOPS_TYPE_F16>(dtype, rows, cols, src, lds, dst, ldd, s);
    return launch_convert_to<REPOPS_TYPE_BF16>(dtype, rows, cols, src, lds, dst, ldd, s);
}

// Span in bytes of a rows x cols operand with pitch ld and element size sz.
bool span_bytes(int64_t rows, int64_t cols, int64_t ld, unsigned sz, uint64_t *out) {
    if (rows == 0 || cols == 0) { *out = 0; return true; }
    if (rows - 1 > (INT64_MAX / 4 - cols) / std::max<int64_t>(ld, 1)) return false;
    *out = uint64_t((rows - 1) * ld + cols) * sz;
    return true;
}

// ---------------------------------------------------------- rolling hash ----

constexpr int ROLL_CHUNK = 64;   // window starts per thread
static_assert(REPOPS_ROLLING_HASH_BASE == roll61::BASE, "roll61 specialises the products by B = 2^32 + 15");

__global__ void __launch_bounds__(256)
rolling_hash_kernel(int64_t rows, int64_t width, const uint32_t *__restrict__ words, int64_t ldw, int64_t W,
                    uint64_t base_w, uint64_t *__restrict__ out, int64_t ldo, int64_t chunks) {
    const int64_t n = width - W + 1;
    const int64_t total = rows * chunks;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < total; t += stride) {
        const int64_t r = t / chunks, c = t - r * chunks;
        const int64_t i0 = c * ROLL_CHUNK, i1 = min(i0 + ROLL_CHUNK, n);
        const uint32_t *w = words + r * ldw;
        uint64_t *o = out + r * ldo;
        uint64_t h = 0;
        for (int64_t k = 0; k < W; ++k) h = roll61::push(h, w[i0 + k]);
        o[i0] = h;
        for (int64_t i = i0 + 1; i < i1; ++i) {
            h = roll61::slide(h, w[i - 1], w[i + W - 1], base_w);
            o[i] = h;
        }
    }
}

// Shared-memory staging: a warp takes SEG = 32 * ROLL_CHUNK consecutive window
// starts of one row and copies the SEG + W - 1 words they read with coalesced
// loads; lane L then rolls over starts 64L .. 64L + 63 reading the stage.  The
// word stage puts one pad slot after every 64 (index j at j + j/64): lane L's
// word k sits at 65L + k + k/64, so the 32 lanes hit 32 different banks.  The
// hashes leave ROLL_GROUP steps at a time through a small second stage (row L
// holds lane L's last ROLL_GROUP hashes, rows padded to an odd count of
// 8-byte slots): each 8-byte store instruction then writes four runs of 64
// contiguous bytes.  64 starts a lane halve the share of Horner's rule at
// window 32; blocks of 4 warps then still fit 5 to an SM.
constexpr int ROLL_SEG = 32 * ROLL_CHUNK;
constexpr int ROLL_WARPS = 4;
constexpr int ROLL_GROUP = 8;                              // steps per output copy
constexpr int ROLL_OROW = ROLL_GROUP + 1;                  // 8-byte slots per stage row
constexpr int ROLL_OSTAGE = 32 * ROLL_OROW;                // 8-byte slots per warp
constexpr int64_t ROLL_MAX_STAGED_WINDOW = 1024;
static_assert(ROLL_CHUNK % ROLL_GROUP == 0, "whole groups");

__device__ __forceinline__ int padded(int j) { return j + j / ROLL_CHUNK; }

__global__ void __launch_bounds__(32 * ROLL_WARPS)
rolling_hash_staged_kernel(int64_t rows, int64_t width, const uint32_t *__restrict__ words, int64_t ldw, int W,
                           uint64_t base_w, uint64_t *__restrict__ out, int64_t ldo, int64_t segs) {
    extern __shared__ uint64_t roll_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wcap = padded(ROLL_SEG + W - 1) + 1;                       // words per warp stage
    uint64_t *ostage = roll_smem + warp * ROLL_OSTAGE;
    uint32_t *wstage = reinterpret_cast<uint32_t *>(roll_smem + ROLL_WARPS * ROLL_OSTAGE) + warp * wcap;
    const int64_t n = width - W + 1;
    const int64_t total = rows * segs;
    for (int64_t t = int64_t(blockIdx.x) * ROLL_WARPS + warp; t < total; t += int64_t(gridDim.x) * ROLL_WARPS) {
        const int64_t r = t / segs, s0 = (t - r * segs) * ROLL_SEG;
        const uint32_t *w = words + r * ldw + s0;
        const int nw = int(min(int64_t(ROLL_SEG + W - 1), width - s0));   // words of this segment
        for (int j = lane; j < nw; j += 32) wstage[padded(j)] = __ldcs(w + j);
        __syncwarp();
        const int i0 = lane * ROLL_CHUNK;                                // local start of this lane
        const int cnt = int(max(int64_t(0), min(int64_t(ROLL_CHUNK), n - s0 - i0)));
        const int nout = int(min(int64_t(ROLL_SEG), n - s0));            // hashes of this segment
        uint64_t *o = out + r * ldo + s0;
        uint64_t h = 0;
        if (cnt > 0)
            for (int k = 0; k < W; ++k) h = roll61::push(h, wstage[padded(i0 + k)]);
        for (int g = 0; g < ROLL_CHUNK && g < nout; g += ROLL_GROUP) {   // lane 0 holds start g
#pragma unroll
            for (int k = 0; k < ROLL_GROUP; ++k) {
                const int i = g + k;
                if (i > 0 && i < cnt)
                    h = roll61::slide(h, wstage[padded(i0 + i - 1)], wstage[padded(i0 + i + W - 1)], base_w);
                ostage[lane * ROLL_OROW + k] = h;                        // slots past cnt are never copied
            }
            __syncwarp();
            // slot q*32 + lane: row (lane L' = its 8-slot run) and step within the group
#pragma unroll
            for (int q = 0; q < ROLL_GROUP; ++q) {
                const int idx = q * 32 + lane, row = idx / ROLL_GROUP, k = idx % ROLL_GROUP;
                const int j = row * ROLL_CHUNK + g + k;                  // local window start
                if (j < nout) __stcs(o + j, ostage[row * ROLL_OROW + k]);
            }
            __syncwarp();                                                 // stage free for the next group
        }
    }
}

uint64_t powmod61_host(uint64_t b, int64_t e) {
    unsigned __int128 r = 1, x = b % roll61::P;
    while (e > 0) {
        if (e & 1) r = (r * x) % roll61::P;
        x = (x * x) % roll61::P;
        e >>= 1;
    }
    return uint64_t(r);
}

}  // namespace
}  // namespace repops

using namespace repops;

extern "C" int repops_gemm_f32_config(int config, int loader, int transA, int transB, int64_t M, int64_t N,
                                      int64_t K, const float *A, int64_t lda, const float *B, int64_t ldb,
                                      float *C, int64_t ldc, cudaStream_t stream);

extern "C" int repops_convert(int64_t n, const void *src, int src_type, void *dst, int dst_type,
                              cudaStream_t stream) {
    if (n < 0 || !known_type(src_type) || !known_type(dst_type)) return REPOPS_ERR_INVALID_ARG;
    if (n == 0) return REPOPS_OK;
    if (!src || !dst || n > INT64_MAX / 4) return REPOPS_ERR_INVALID_ARG;
    const uint64_t sb = uint64_t(n) * type_size(src_type), db = uint64_t(n) * type_size(dst_type);
    const bool same_place = src == dst && type_size(src_type) == type_size(dst_type);
    if (!same_place && ranges_overlap(src, sb, dst, db)) return REPOPS_ERR_ALIAS;
    if (src_type == dst_type) {
        if (src == dst) return REPOPS_OK;
        cudaError_t e = cudaMemcpyAsync(dst, src, sb, cudaMemcpyDeviceToDevice, stream);
        return e == cudaSuccess ? REPOPS_OK : set_cuda_error(e);
    }
    return launch_convert(src_type, dst_type, 1, n, src, n, dst, n, stream);
}

extern "C" int repops_gemm_typed(int config, int loader, int transA, int transB, int64_t M, int64_t N, int64_t K,
                                 const void *A, int typeA, int64_t lda, const void *B, int typeB, int64_t ldb,
                                 void *C, int typeC, int64_t ldc, cudaStream_t stream) {
    if (!known_type(typeA) || !known_type(typeB) || !known_type(typeC)) return REPOPS_ERR_INVALID_ARG;
    if (typeA == REPOPS_TYPE_F32 && typeB == REPOPS_TYPE_F32 && typeC == REPOPS_TYPE_F32)
        return repops_gemm_f32_config(config, loader, transA, transB, M, N, K, static_cast<const float *>(A), lda,
                                      static_cast<const float *>(B), ldb, static_cast<float *>(C), ldc, stream);
    if (M < 0 || N < 0 || K < 0) return REPOPS_ERR_INVALID_ARG;
    const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;
    if (lda < std::max<int64_t>(1, a_cols) || ldb < std::max<int64_t>(1, b_cols) || ldc < std::max<int64_t>(1, N))
        return REPOPS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return REPOPS_OK;
    if (!C || (K > 0 && (!A || !B))) return REPOPS_ERR_INVALID_ARG;
    uint64_t ab = 0, bb = 0, cb = 0;
    if (!span_bytes(a_rows, a_cols, lda, type_size(typeA), &ab) ||
        !span_bytes(b_rows, b_cols, ldb, type_size(typeB), &bb) || !span_bytes(M, N, ldc, type_size(typeC), &cb))
        return REPOPS_ERR_INVALID_ARG;
    if (ranges_overlap(C, cb, A, ab) || ranges_overlap(C, cb, B, bb)) return REPOPS_ERR_ALIAS;

    // widened copies with a 16-byte pitch (the TMA loader's rule)
    const bool wa = typeA != REPOPS_TYPE_F32 && K > 0, wb = typeB != REPOPS_TYPE_F32 && K > 0;
    const bool wc = typeC != REPOPS_TYPE_F32;
    const int64_t pa = (a_cols + 3) / 4 * 4, pb = (b_cols + 3) / 4 * 4, pc = (N + 3) / 4 * 4;
    const uint64_t na = wa ? uint64_t(a_rows) * pa : 0, nb = wb ? uint64_t(b_rows) * pb : 0;
    const uint64_t nc = wc ? uint64_t(M) * pc : 0;
    void *scratch = nullptr;
    if (scratch_malloc(&scratch, (na + nb + nc) * 4u, stream) != cudaSuccess) {
        cudaGetLastError();
        return REPOPS_ERR_ALLOC;
    }
    float *A32 = static_cast<float *>(scratch), *B32 = A32 + na, *C32 = B32 + nb;
    int rc = REPOPS_OK;
    if (wa) rc = launch_convert(typeA, REPOPS_TYPE_F32, a_rows, a_cols, A, lda, A32, pa, stream);
    if (rc == REPOPS_OK && wb) rc = launch_convert(typeB, REPOPS_TYPE_F32, b_rows, b_cols, B, ldb, B32, pb, stream);
    if (rc == REPOPS_OK)
        rc = repops_gemm_f32_config(config, loader, transA, transB, M, N, K,
                                    wa ? A32 : static_cast<const float *>(A), wa ? pa : lda,
                                    wb ? B32 : static_cast<const float *>(B), wb ? pb : ldb,
                                    wc ? C32 : static_cast<float *>(C), wc ? pc : ldc, stream);
    if (rc == REPOPS_OK && wc) rc = launch_convert(REPOPS_TYPE_F32, typeC, M, N, C32, pc, C, ldc, stream);
    const cudaError_t e = cudaFreeAsync(scratch, stream);
    if (rc == REPOPS_OK && e != cudaSuccess) rc = set_cuda_error(e);
    return rc;
}

extern "C" int repops_rolling_hash_u32(int64_t rows, int64_t width, const uint32_t *words, int64_t ldw,
                                       int64_t window, uint64_t *out, int64_t ldo, cudaStream_t stream) {
    if (rows < 0 || width < 0) return REPOPS_ERR_INVALID_ARG;
    if (rows == 0) return REPOPS_OK;
    if (window < 1 || window > width) return REPOPS_ERR_INVALID_ARG;
    const int64_t n = width - window + 1;
    if (!words || !out || ldw < width || ldo < n) return REPOPS_ERR_INVALID_ARG;
    if (rows - 1 > (INT64_MAX / 8 - width) / ldw || rows - 1 > (INT64_MAX / 8 - n) / ldo)
        return REPOPS_ERR_INVALID_ARG;
    const uint64_t wb = uint64_t((rows - 1) * ldw + width) * 4u, ob = uint64_t((rows - 1) * ldo + n) * 8u;
    if (ranges_overlap(words, wb, out, ob)) return REPOPS_ERR_ALIAS;
    DeviceInfo di;
    const int sms = current_device_info(&di) == REPOPS_OK ? di.sms : 152;
    const uint64_t bw = powmod61_host(REPOPS_ROLLING_HASH_BASE, window);   // B^W mod P
    if (window <= ROLL_MAX_STAGED_WINDOW) {
        const int64_t segs = (n + ROLL_SEG - 1) / ROLL_SEG;
        const int wcap = int(ROLL_SEG + window - 1) + int((ROLL_SEG + window - 1) / ROLL_CHUNK) + 1;
        const size_t smem = size_t(ROLL_WARPS) * (size_t(ROLL_OSTAGE) * 8u + size_t(wcap) * 4u);
        cudaError_t e = cudaFuncSetAttribute(rolling_hash_staged_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return set_cuda_error(e);
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rolling_hash_staged_kernel, 32 * ROLL_WARPS, smem);
        if (e != cudaSuccess) return set_cuda_error(e);
        const int blocks = int(std::min<int64_t>((rows * segs + ROLL_WARPS - 1) / ROLL_WARPS,
                                                 int64_t(std::max(per_sm, 1)) * sms));
        rolling_hash_staged_kernel<<<blocks, 32 * ROLL_WARPS, smem, stream>>>(
            rows, width, words, ldw, int(window), bw, out, ldo, segs);
        return check_launch();
    }
    const int64_t chunks = (n + ROLL_CHUNK - 1) / ROLL_CHUNK;
    const int blocks = int(std::min<int64_t>((rows * chunks + 255) / 256, int64_t(sms) * 16));
    rolling_hash_kernel<<<blocks, 256, 0, stream>>>(rows, width, words, ldw, window, bw, out, ldo, chunks);
    return check_launch();
}
