// gemm_kernels.cuh -- the order-fixed FP32 GEMM kernels (SIMT, sm_103a).
//
// What is computed ("Verde与RepOps" §3.2, matmul example): for every output
// element, sum = +0; for k = 0 .. K-1 in increasing order: sum = fl(sum +
// fl(A[i][k] * B[k][j])).  The product and the add are separate IEEE
// round-to-nearest operations (__fmul_rn / __fadd_rn are never contracted into
// a fused multiply-add; the library is also built with -fmad=false).  Tensor
// cores are not used: their internal accumulation order and rounding would
// change the bits.
//
// How it is parallelised (§3.2 design principle: order-independent dimensions
// run in parallel, the order-critical one runs serially):
//   - each CTA owns a BM x BN tile of C, each thread a TM x TN sub-tile held in
//     registers; the k loop is the only serial loop and every accumulator sees
//     k = 0, 1, 2, ... in that order -- no split-K, no reassociation;
//   - operands are staged through a STAGES-deep shared-memory ring of BK = 32
//     k-slices, filled either by TMA (cp.async.bulk.tensor, one elected thread,
//     completion on an mbarrier) or, for operands TMA cannot describe
//     (unaligned pointers or leading dimensions), by 4-byte cp.async with zero
//     fill.  Both loaders produce the same shared-memory image;
//   - the k tail is zero-filled in BOTH operands.  fl(0*0) = +0, and the
//     accumulator is never -0 (it starts at +0, and round-to-nearest gives +0
//     for an exact cancellation), so adding +0 leaves it bit-identical.
//
// Shared-memory layouts of one stage:
//   K-inner operand (A stored row-major, or B stored transposed): [rows][32]
//     fp32, 128-byte rows, with the TMA 128-byte swizzle -- 16-byte chunk c of
//     row r sits at chunk c ^ (r mod 8).  A thread reads a float4 along k.
//   MN-inner operand (A stored transposed, or B row-major): [32][rows] plain.
//     A thread reads float4 runs along m or n.
// Within a warp the 32 lanes form a 4 (m) x 8 (n) grid.  Lanes that share m
// read the same A address (broadcast); the n mapping is chosen per B layout so
// that each quarter-warp's B reads hit 8 distinct 16-byte bank groups:
//   B MN-inner: lane ln owns columns ln*4 + 32*q + {0..3}  (128 contiguous bytes)
//   B K-inner : lane ln owns columns ln + 8*c              (distinct swizzle rows)
#pragma once

#include "gemm_common.h"
#include "internal.cuh"

namespace repops {
namespace gemm {

constexpr int BK = 32;   // k-extent of one stage: 32 fp32 = one 128-byte row

template <int TM_, int TN_, int WARPS_M_, int WARPS_N_, int STAGES_>
struct Tile {
    static constexpr int TM = TM_, TN = TN_;
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_, STAGES = STAGES_;
    static constexpr int WM = 4 * TM, WN = 8 * TN;   // warp tile: 4 x 8 lanes
    static constexpr int BM = WARPS_M * WM, BN = WARPS_N * WN;
    static constexpr int THREADS = 32 * WARPS_M * WARPS_N;
    static constexpr int A_FLOATS = BM * BK, B_FLOATS = BN * BK;
    static constexpr int STAGE_FLOATS = A_FLOATS + B_FLOATS;
    static constexpr int STAGE_BYTES = STAGE_FLOATS * 4;
    // ring + 1 KiB for aligning the base to the 1 KiB swizzle atom + barriers
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 8 * STAGES;
    static_assert(TM % 4 == 0 && TN % 4 == 0, "per-thread tile is made of float4 runs");
    static_assert(BM % 8 == 0 && BN % 8 == 0, "the swizzle atom is 8 rows");
    static_assert(BM <= 256 && BN <= 256, "TMA box extent is at most 256");
};

// Float offset of element (r, k) in a K-inner [rows][32] tile with the TMA
// 128-byte swizzle (tile base aligned to 1 KiB).
__device__ __forceinline__ int kin_off(int r, int k) {
    return r * BK + ((((k >> 2) ^ (r & 7)) << 2) | (k & 3));
}

// Grouped rasterisation: consecutive CTAs walk down GROUP tile-rows before
// moving right, so CTAs resident together share A row-panels and B column-panels
// in L2.
__device__ __forceinline__ void tile_coords(int bid, int tiles_m, int tiles_n, int &tm, int &tn) {
    constexpr int GROUP = 8;
    const int per_group = GROUP * tiles_n;
    const int g = bid / per_group;
    const int first_m = g * GROUP;
    const int gm = min(tiles_m - first_m, GROUP);
    const int in_group = bid - g * per_group;
    tm = first_m + in_group % gm;
    tn = in_group / gm;
}

// Row of the CTA tile held in a thread's accumulator row r.
//   A K-inner:  abase + 4r   (abase = warp row base + lm): rows of one thread
//               have swizzle key lm or lm^4, so one XOR per k-chunk serves all.
//   A MN-inner: abase + r    (abase = warp row base + lm*TM): float4 runs in m.
template <bool A_KIN>
__device__ __forceinline__ int a_row(int abase, int r) { return A_KIN ? abase + 4 * r : abase + r; }

// Column of the CTA tile held in a thread's accumulator column c.
//   B K-inner:  bbase + 8c   (bbase = warp col base + ln): swizzle key ln.
//   B MN-inner: bbase + 32*(c/4) + c%4  (bbase = warp col base + 4*ln).
template <bool B_KIN>
__device__ __forceinline__ int b_col(int bbase, int c) {
    return B_KIN ? bbase + 8 * c : bbase + 32 * (c / 4) + (c % 4);
}

// One stage (32 k-steps) of the serial k-chain for this thread's TM x TN
// accumulators.  k advances in increasing order: k4 (chunks of 4), then kk.
template <class T, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void mma_stage(const float *__restrict__ As, const float *__restrict__ Bs,
                                          int abase, int bbase, int lm, int ln,
                                          float (&acc)[T::TM][T::TN]) {
#pragma unroll 2
    for (int k4 = 0; k4 < BK / 4; ++k4) {
        float a[T::TM][4];
        float b[T::TN][4];
        if constexpr (A_KIN) {
            // rows abase + 4r: swizzle key lm for even r, lm ^ 4 for odd r
            const int t0 = (k4 ^ lm) << 2;
            const float *p0 = As + abase * BK + t0;
            const float *p1 = As + abase * BK + (t0 ^ 16);
#pragma unroll
            for (int r = 0; r < T::TM; ++r) {
                const float4 v = *reinterpret_cast<const float4 *>(((r & 1) ? p1 : p0) + r * 4 * BK);
                a[r][0] = v.x; a[r][1] = v.y; a[r][2] = v.z; a[r][3] = v.w;
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int q = 0; q < T::TM / 4; ++q) {
                    const float4 v = *reinterpret_cast<const float4 *>(
                        As + (4 * k4 + kk) * T::BM + abase + 4 * q);
                    a[4 * q + 0][kk] = v.x; a[4 * q + 1][kk] = v.y;
                    a[4 * q + 2][kk] = v.z; a[4 * q + 3][kk] = v.w;
                }
            }
        }
        if constexpr (B_KIN) {
            // columns bbase + 8c all have swizzle key ln
            const float *bp = Bs + bbase * BK + ((k4 ^ ln) << 2);
#pragma unroll
            for (int c = 0; c < T::TN; ++c) {
                const float4 v = *reinterpret_cast<const float4 *>(bp + c * 8 * BK);
                b[c][0] = v.x; b[c][1] = v.y; b[c][2] = v.z; b[c][3] = v.w;
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int q = 0; q < T::TN / 4; ++q) {
                    const float4 v = *reinterpret_cast<const float4 *>(
                        Bs + (4 * k4 + kk) * T::BN + bbase + 32 * q);
                    b[4 * q + 0][kk] = v.x; b[4 * q + 1][kk] = v.y;
                    b[4 * q + 2][kk] = v.z; b[4 * q + 3][kk] = v.w;
                }
            }
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int r = 0; r < T::TM; ++r) {
#pragma unroll
                for (int c = 0; c < T::TN; ++c) {
                    acc[r][c] = __fadd_rn(acc[r][c], __fmul_rn(a[r][kk], b[c][kk]));
                }
            }
        }
    }
}

// Writes the thread's accumulators; rows/columns past M/N are skipped.
template <class T, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void store_tile(float *__restrict__ C, int64_t ldc, int64_t M, int64_t N,
                                           int64_t m0, int64_t n0, int abase, int bbase,
                                           const float (&acc)[T::TM][T::TN], bool c_vec) {
#pragma unroll
    for (int r = 0; r < T::TM; ++r) {
        const int64_t gm = m0 + a_row<A_KIN>(abase, r);
        if (gm >= M) break;   // rows increase with r
        float *crow = C + gm * ldc;
        if constexpr (!B_KIN) {
#pragma unroll
            for (int q = 0; q < T::TN / 4; ++q) {
                const int64_t gn = n0 + bbase + 32 * q;
                if (c_vec && gn + 3 < N) {
                    *reinterpret_cast<float4 *>(crow + gn) =
                        make_float4(acc[r][4 * q], acc[r][4 * q + 1], acc[r][4 * q + 2], acc[r][4 * q + 3]);
                } else {
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (gn + t < N) crow[gn + t] = acc[r][4 * q + t];
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < T::TN; ++c) {
                const int64_t gn = n0 + b_col<true>(bbase, c);
                if (gn < N) crow[gn] = acc[r][c];
            }
        }
    }
}

template <class T>
__device__ __forceinline__ float *aligned_smem_base(unsigned char *raw) {
    return reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------------ TMA ----

template <class T, bool A_KIN, bool B_KIN>
__global__ void __launch_bounds__(T::THREADS, 1)
gemm_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                float *__restrict__ C, int64_t M, int64_t N, int64_t K, int64_t ldc,
                int tiles_m, int tiles_n, int c_vec, unsigned *status) {
    extern __shared__ unsigned char smem_raw[];
    float *smem = aligned_smem_base<T>(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + T::STAGES * T::STAGE_FLOATS);

    const int tid = threadIdx.x;
    int tm, tn;
    tile_coords(blockIdx.x, tiles_m, tiles_n, tm, tn);
    const int64_t m0 = int64_t(tm) * T::BM, n0 = int64_t(tn) * T::BN;
    const int KT = int((K + BK - 1) / BK);

    if (tid == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
#pragma unroll 1
        for (int s = 0; s < T::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncthreads();

    // thread 0 only: put k-slice `kt` in flight into its ring slot
    auto issue = [&](int kt) {
        const int s = kt % T::STAGES;
        float *As = smem + s * T::STAGE_FLOATS;
        float *Bs = As + T::A_FLOATS;
        mbar_arrive_expect_tx(&bars[s], T::STAGE_BYTES);
        const int k0 = kt * BK;
        if constexpr (A_KIN) tma_load_2d(As, &tmA, &bars[s], k0, int(m0));
        else                 tma_load_2d(As, &tmA, &bars[s], int(m0), k0);
        if constexpr (B_KIN) tma_load_2d(Bs, &tmB, &bars[s], k0, int(n0));
        else                 tma_load_2d(Bs, &tmB, &bars[s], int(n0), k0);
    };

    int issued = 0;
    if (tid == 0) {
#pragma unroll 1
        for (; issued < T::STAGES - 1 && issued < KT; ++issued) issue(issued);
    }

    const int warp = tid >> 5, lane = tid & 31;
    const int warp_m = warp % T::WARPS_M, warp_n = warp / T::WARPS_M;
    const int lm = lane >> 3, ln = lane & 7;
    const int abase = warp_m * T::WM + (A_KIN ? lm : lm * T::TM);
    const int bbase = warp_n * T::WN + (B_KIN ? ln : ln * 4);

    float acc[T::TM][T::TN];
#pragma unroll
    for (int r = 0; r < T::TM; ++r)
#pragma unroll
        for (int c = 0; c < T::TN; ++c) acc[r][c] = 0.0f;

    int bail = 0;
#pragma unroll 1
    for (int kt = 0; kt < KT; ++kt) {
        // every thread is done with the slot consumed in iteration kt-1
        if (__syncthreads_or(bail)) { bail = 1; break; }
        if (tid == 0 && issued < KT) { issue(issued); ++issued; }
        const int s = kt % T::STAGES;
        if (!mbar_wait_bounded(&bars[s], uint32_t(kt / T::STAGES) & 1u)) { bail = 1; continue; }
        const float *As = smem + s * T::STAGE_FLOATS;
        mma_stage<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, abase, bbase, lm, ln, acc);
    }
    if (__syncthreads_or(bail)) {
        if (tid == 0) {
            atomicOr(status, 1u);
            // let this CTA's copies still in flight land before it exits
#pragma unroll 1
            for (int kt = max(0, issued - T::STAGES); kt < issued; ++kt)
                mbar_wait_bounded(&bars[kt % T::STAGES], uint32_t(kt / T::STAGES) & 1u);
        }
        return;
    }
    store_tile<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec != 0);
}

// ------------------------------------------------------------- cp.async ----

// Fills one ring slot with k-slice [k0, k0 + 32) of both operands, 4 bytes per
// copy, zero-filling everything outside the matrices.
template <class T, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void load_slice_cpasync(float *As, float *Bs, const float *__restrict__ A,
                                                   int64_t lda, const float *__restrict__ B, int64_t ldb,
                                                   int64_t M, int64_t N, int64_t K,
                                                   int64_t m0, int64_t n0, int64_t k0, int tid) {
    constexpr int NW = T::THREADS / 32;
    if constexpr (A_KIN) {
        // element (r, k): a warp copies one 128-byte row segment
        const int k = tid & 31;
        const int64_t gk = k0 + k;
#pragma unroll 4
        for (int r = tid >> 5; r < T::BM; r += NW) {
            const int64_t gm = m0 + r;
            const bool ok = gk < K && gm < M;
            cp_async_4(As + kin_off(r, k), ok ? A + gm * lda + gk : A, ok ? 4u : 0u);
        }
    } else {
#pragma unroll 4
        for (int e = tid; e < BK * T::BM; e += T::THREADS) {
            const int k = e / T::BM, r = e % T::BM;
            const int64_t gk = k0 + k, gm = m0 + r;
            const bool ok = gk < K && gm < M;
            cp_async_4(As + k * T::BM + r, ok ? A + gk * lda + gm : A, ok ? 4u : 0u);
        }
    }
    if constexpr (B_KIN) {
        const int k = tid & 31;
        const int64_t gk = k0 + k;
#pragma unroll 4
        for (int r = tid >> 5; r < T::BN; r += NW) {
            const int64_t gn = n0 + r;
            const bool ok = gk < K && gn < N;
            cp_async_4(Bs + kin_off(r, k), ok ? B + gn * ldb + gk : B, ok ? 4u : 0u);
        }
    } else {
#pragma unroll 4
        for (int e = tid; e < BK * T::BN; e += T::THREADS) {
            const int k = e / T::BN, r = e % T::BN;
            const int64_t gk = k0 + k, gn = n0 + r;
            const bool ok = gk < K && gn < N;
            cp_async_4(Bs + k * T::BN + r, ok ? B + gk * ldb + gn : B, ok ? 4u : 0u);
        }
    }
}

template <class T, bool A_KIN, bool B_KIN>
__global__ void __launch_bounds__(T::THREADS, 1)
gemm_cpasync_kernel(const float *__restrict__ A, int64_t lda, const float *__restrict__ B, int64_t ldb,
                    float *__restrict__ C, int64_t M, int64_t N, int64_t K, int64_t ldc,
                    int tiles_m, int tiles_n, int c_vec) {
    extern __shared__ unsigned char smem_raw[];
    float *smem = aligned_smem_base<T>(smem_raw);

    const int tid = threadIdx.x;
    int tm, tn;
    tile_coords(blockIdx.x, tiles_m, tiles_n, tm, tn);
    const int64_t m0 = int64_t(tm) * T::BM, n0 = int64_t(tn) * T::BN;
    const int KT = int((K + BK - 1) / BK);

#pragma unroll 1
    for (int s = 0; s < T::STAGES - 1; ++s) {
        if (s < KT) {
            float *As = smem + s * T::STAGE_FLOATS;
            load_slice_cpasync<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, A, lda, B, ldb, M, N, K,
                                                m0, n0, int64_t(s) * BK, tid);
        }
        cp_async_commit();
    }

    const int warp = tid >> 5, lane = tid & 31;
    const int warp_m = warp % T::WARPS_M, warp_n = warp / T::WARPS_M;
    const int lm = lane >> 3, ln = lane & 7;
    const int abase = warp_m * T::WM + (A_KIN ? lm : lm * T::TM);
    const int bbase = warp_n * T::WN + (B_KIN ? ln : ln * 4);

    float acc[T::TM][T::TN];
#pragma unroll
    for (int r = 0; r < T::TM; ++r)
#pragma unroll
        for (int c = 0; c < T::TN; ++c) acc[r][c] = 0.0f;

#pragma unroll 1
    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<T::STAGES - 2>();   // slice kt has landed (this thread's copies)
        __syncthreads();                  // ... and everyone's; slot kt-1 is free
        const int nk = kt + T::STAGES - 1;
        if (nk < KT) {
            float *As = smem + (nk % T::STAGES) * T::STAGE_FLOATS;
            load_slice_cpasync<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, A, lda, B, ldb, M, N, K,
                                                m0, n0, int64_t(nk) * BK, tid);
        }
        cp_async_commit();
        const float *As = smem + (kt % T::STAGES) * T::STAGE_FLOATS;
        mma_stage<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, abase, bbase, lm, ln, acc);
    }
    cp_async_wait<0>();
    store_tile<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec != 0);
}

// --------------------------------------------------------------- host ----

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (null when unavailable).
EncodeTiledFn tensor_map_encoder();

// 2-D fp32 tensor map: inner extent `inner`, outer extent `outer`, row pitch
// `ld` elements, box (box_inner x box_outer), zero fill out of bounds.
inline bool make_map(CUtensorMap *map, const float *base, int64_t inner, int64_t outer, int64_t ld,
                     int box_inner, int box_outer, bool swizzle128) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    cuuint64_t strides[1] = {cuuint64_t(ld) * 4u};
    cuuint32_t box[2] = {cuuint32_t(box_inner), cuuint32_t(box_outer)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <class T, bool A_KIN, bool B_KIN>
int launch_tma(const GemmProblem &p, int tiles_m, int tiles_n, int c_vec) {
    CUtensorMap ma, mb;
    // A: row-major (K-inner) -> dims {K, M}; transposed (M-inner) -> {M, K}
    const bool okA = A_KIN ? make_map(&ma, p.A, p.K, p.M, p.lda, BK, T::BM, true)
                           : make_map(&ma, p.A, p.M, p.K, p.lda, T::BM, BK, false);
    // B: transposed (K-inner) -> dims {K, N}; row-major (N-inner) -> {N, K}
    const bool okB = B_KIN ? make_map(&mb, p.B, p.K, p.N, p.ldb, BK, T::BN, true)
                           : make_map(&mb, p.B, p.N, p.K, p.ldb, T::BN, BK, false);
    if (!okA || !okB) return REPOPS_ERR_UNSUPPORTED;
    auto kern = gemm_tma_kernel<T, A_KIN, B_KIN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return set_cuda_error(e);
    kern<<<tiles_m * tiles_n, T::THREADS, T::SMEM_BYTES, p.stream>>>(
        ma, mb, p.C, p.M, p.N, p.K, p.ldc, tiles_m, tiles_n, c_vec, p.status);
    return check_launch();
}

template <class T, bool A_KIN, bool B_KIN>
int launch_cpasync(const GemmProblem &p, int tiles_m, int tiles_n, int c_vec) {
    auto kern = gemm_cpasync_kernel<T, A_KIN, B_KIN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return set_cuda_error(e);
    kern<<<tiles_m * tiles_n, T::THREADS, T::SMEM_BYTES, p.stream>>>(
        p.A, p.lda, p.B, p.ldb, p.C, p.M, p.N, p.K, p.ldc, tiles_m, tiles_n, c_vec);
    return check_launch();
}

// loader: REPOPS_LOADER_TMA or REPOPS_LOADER_CPASYNC (already resolved).
template <class T>
int launch_config(const GemmProblem &p, int loader) {
    const int64_t tiles_m = (p.M + T::BM - 1) / T::BM;
    const int64_t tiles_n = (p.N + T::BN - 1) / T::BN;
    if (tiles_m * tiles_n > 0x7fffffffLL) return REPOPS_ERR_UNSUPPORTED;
    const int c_vec = (reinterpret_cast<uintptr_t>(p.C) % 16 == 0) && (p.ldc % 4 == 0);
    const bool a_kin = p.transA == 0, b_kin = p.transB != 0;
    const int tmi = int(tiles_m), tni = int(tiles_n);
    if (loader == REPOPS_LOADER_TMA) {
        if (a_kin && !b_kin) return launch_tma<T, true, false>(p, tmi, tni, c_vec);
        if (a_kin && b_kin) return launch_tma<T, true, true>(p, tmi, tni, c_vec);
        if (!a_kin && !b_kin) return launch_tma<T, false, false>(p, tmi, tni, c_vec);
        return launch_tma<T, false, true>(p, tmi, tni, c_vec);
    }
    if (a_kin && !b_kin) return launch_cpasync<T, true, false>(p, tmi, tni, c_vec);
    if (a_kin && b_kin) return launch_cpasync<T, true, true>(p, tmi, tni, c_vec);
    if (!a_kin && !b_kin) return launch_cpasync<T, false, false>(p, tmi, tni, c_vec);
    return launch_cpasync<T, false, true>(p, tmi, tni, c_vec);
}

template <class T>
int occupancy() {
    auto kern = gemm_tma_kernel<T, true, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, T::THREADS, T::SMEM_BYTES) != cudaSuccess)
        return 0;
    return n;
}

template <class T>
GemmConfigInfo info() {
    return GemmConfigInfo{T::BM, T::BN, T::THREADS, T::TM, T::TN, T::STAGES};
}

}  // namespace gemm
}  // namespace repops

// Defines the three entry points of one configuration.
#define REPOPS_DEFINE_GEMM_CONFIG(N, TILE)                                                        \
    namespace repops {                                                                            \
    int gemm_launch_cfg##N(const GemmProblem &p, int loader) { return gemm::launch_config<TILE>(p, loader); } \
    int gemm_occupancy_cfg##N() { return gemm::occupancy<TILE>(); }                               \
    GemmConfigInfo gemm_info_cfg##N() { return gemm::info<TILE>(); }                              \
    }
