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
// takes 16 consecutive window starts of one row: Horner's rule for the first,
// then h' = (h - w_out * B^(W-1)) * B + w_in for the rest -- exact modular
// integers, so the split of a row across threads does not change a bit.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"

namespace repops {
namespace {

bool known_type(int t) { return t == REPOPS_TYPE_F32 || t == REPOPS_TYPE_F16 || t == REPOPS_TYPE_BF16; }
unsigned type_size(int t) { return t == REPOPS_TYPE_F32 ? 4u : 2u; }

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

// rows x cols elements: source element (r, c) at src[r*lds + c], destination at
// dst[r*ldd + c] (a 1-D conversion is one row).  Each thread handles the same
// element of source and destination, so an in-place conversion between types
// of one size is safe.
template <int S, int D>
__global__ void __launch_bounds__(256)
convert_kernel(int64_t rows, int64_t cols, const void *src, int64_t lds, void *dst, int64_t ldd) {
    const int64_t total = rows * cols;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += stride) {
        const int64_t r = e / cols, c = e - r * cols;
        store_from_f32<D>(dst, r * ldd + c, load_f32<S>(src, r * lds + c));
    }
}

template <int S>
int launch_convert_to(int dtype, int64_t rows, int64_t cols, const void *src, int64_t lds, void *dst,
                      int64_t ldd, cudaStream_t s) {
    DeviceInfo di;
    const int sms = current_device_info(&di) == REPOPS_OK ? di.sms : 152;
    const int64_t total = rows * cols;
    const int blocks = int(std::min<int64_t>((total + 255) / 256, int64_t(sms) * 16));
    if (dtype == REPOPS_TYPE_F32)
        convert_kernel<S, REPOPS_TYPE_F32><<<blocks, 256, 0, s>>>(rows, cols, src, lds, dst, ldd);
    else if (dtype == REPOPS_TYPE_F16)
        convert_kernel<S, REPOPS_TYPE_F16><<<blocks, 256, 0, s>>>(rows, cols, src, lds, dst, ldd);
    else
        convert_kernel<S, REPOPS_TYPE_BF16><<<blocks, 256, 0, s>>>(rows, cols, src, lds, dst, ldd);
    return check_launch();
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

constexpr uint64_t P61 = (uint64_t(1) << 61) - 1;
constexpr int ROLL_CHUNK = 16;   // window starts per thread

__device__ __forceinline__ uint64_t mulmod61(uint64_t a, uint64_t b) {
    // a, b < 2^61: a*b = hi*2^64 + lo, and 2^64 = 8 * 2^61 = 8 (mod P), so
    // a*b = (lo & P) + (lo >> 61) + 8*hi (mod P); 8*hi < 2^61 leaves the low
    // three bits free for lo >> 61
    const uint64_t lo = a * b, hi = __umul64hi(a, b);
    uint64_t r = (lo & P61) + ((lo >> 61) | (hi << 3));   // < 2^62
    r = (r & P61) + (r >> 61);                              // <= P + 1
    return r >= P61 ? r - P61 : r;
}

__device__ __forceinline__ uint64_t addmod61(uint64_t a, uint64_t b) {   // a, b < P
    const uint64_t s = a + b;
    return s >= P61 ? s - P61 : s;
}

__global__ void __launch_bounds__(256)
rolling_hash_kernel(int64_t rows, int64_t width, const uint32_t *__restrict__ words, int64_t ldw, int64_t W,
                    uint64_t base, uint64_t base_w1, uint64_t *__restrict__ out, int64_t ldo, int64_t chunks) {
    const int64_t n = width - W + 1;
    const int64_t total = rows * chunks;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < total; t += stride) {
        const int64_t r = t / chunks, c = t - r * chunks;
        const int64_t i0 = c * ROLL_CHUNK, i1 = min(i0 + ROLL_CHUNK, n);
        const uint32_t *w = words + r * ldw;
        uint64_t *o = out + r * ldo;
        uint64_t h = 0;
        for (int64_t k = 0; k < W; ++k) h = addmod61(mulmod61(h, base), w[i0 + k]);
        o[i0] = h;
        for (int64_t i = i0 + 1; i < i1; ++i) {
            const uint64_t drop = mulmod61(w[i - 1], base_w1);
            h = h >= drop ? h - drop : h + (P61 - drop);
            h = addmod61(mulmod61(h, base), w[i + W - 1]);
            o[i] = h;
        }
    }
}

uint64_t powmod61_host(uint64_t b, int64_t e) {
    unsigned __int128 r = 1, x = b % P61;
    while (e > 0) {
        if (e & 1) r = (r * x) % P61;
        x = (x * x) % P61;
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
    if (cudaMallocAsync(&scratch, (na + nb + nc) * 4u, stream) != cudaSuccess) {
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
    const int64_t chunks = (n + ROLL_CHUNK - 1) / ROLL_CHUNK;
    DeviceInfo di;
    const int sms = current_device_info(&di) == REPOPS_OK ? di.sms : 152;
    const int blocks = int(std::min<int64_t>((rows * chunks + 255) / 256, int64_t(sms) * 16));
    rolling_hash_kernel<<<blocks, 256, 0, stream>>>(rows, width, words, ldw, window, REPOPS_ROLLING_HASH_BASE,
                                                    powmod61_host(REPOPS_ROLLING_HASH_BASE, window - 1), out, ldo,
                                                    chunks);
    return check_launch();
}
