// gemm_kernels.cuh -- the order-fixed FP32 GEMM kernels (SIMT, sm_103a).
//
// What is computed ("Verde与RepOps" §3.2, matmul example): for every output
// element, sum = +0; for k = 0 .. K-1 in increasing order: sum = fl(sum +
// fl(A[i][k] * B[k][j])).  The product and the add are separate IEEE
// round-to-nearest operations: products are __fmul_rn (never contracted into a
// fused multiply-add), sums are add.rn.f32x2 -- two independent binary32 adds
// in one instruction, each rounded on its own -- and the library is built with
// -fmad=false.  Tensor cores are not used: their internal accumulation order
// and rounding would change the bits.
//
// How it is parallelised (§3.2 design principle: order-independent dimensions
// run in parallel, the order-critical one runs serially):
//   - each CTA owns a BM x BN tile of C, each thread a TM x TN sub-tile held in
//     registers; the k loop is the only serial loop and every accumulator sees
//     k = 0, 1, 2, ... in that order -- no split-K, no reassociation;
//   - operands are staged through a STAGES-deep shared-memory ring of BK = 32
//     k-slices.  TMA path: a producer warp issues cp.async.bulk.tensor copies,
//     completion is counted on a "full" mbarrier per slot, consumer warps
//     release a slot on its "empty" mbarrier -- no CTA-wide barrier in the main
//     loop.  cp.async path (operands TMA cannot describe: unaligned pointers or
//     leading dimensions): every thread copies 4-byte elements with zero fill.
//     Both loaders produce the same shared-memory image;
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
// Batched / fused-epilogue variant (EX = true): blockIdx.y is the batch; every
// operand advances by its own stride (TMA: a 3-D tensor map whose third
// dimension is the batch, so out-of-bounds zero fill stays per batch).  After
// an element's whole k-chain the epilogue applies y = fl(alpha*acc), then
// fl(y + bias[j]), then GeLU, then fl(y + R[i][j]), each part optional.
//
// Within a warp the 32 lanes form a 4 (m) x 8 (n) grid.  Lanes that share m
// read the same A address (broadcast); the n mapping is chosen per B layout so
// that each quarter-warp's B reads hit 8 distinct 16-byte bank groups:
//   B MN-inner: lane ln owns columns ln*4 + 32*q + {0..3}  (128 contiguous bytes)
//   B K-inner : lane ln owns columns ln + 8*c              (distinct swizzle rows)
#pragma once

#include "fixed_math.cuh"
#include "packed_f32.cuh"
#include "gemm_common.h"
#include "internal.cuh"

namespace repops {
namespace gemm {

constexpr int BK = 32;   // k-extent of one stage: 32 fp32 = one 128-byte row

// Unroll of the 4-k chunk loop inside one 32-k slice.  Measured at 8192^3:
// both operands K-inner run best at 1, every other layout at 4.
template <bool A_KIN, bool B_KIN>
struct K4Unroll {
    static constexpr int value = (A_KIN && B_KIN) ? 1 : 4;
};

// TM x TN accumulators per thread, WARPS_M x WARPS_N consumer warps, STAGES
// ring slots.  MINB_: CTAs per SM the register allocation must allow (0 means
// 2 for CTAs of at most 128 consumer threads, else 1).
template <int TM_, int TN_, int WARPS_M_, int WARPS_N_, int STAGES_, int MINB_ = 0>
struct Tile {
    static constexpr int TM = TM_, TN = TN_;
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_, STAGES = STAGES_;
    static constexpr int MINB = MINB_ ? MINB_ : (32 * WARPS_M_ * WARPS_N_ <= 128 ? 2 : 1);
    static constexpr int WM = 4 * TM, WN = 8 * TN;   // warp tile: 4 x 8 lanes
    static constexpr int BM = WARPS_M * WM, BN = WARPS_N * WN;
    static constexpr int THREADS = 32 * WARPS_M * WARPS_N;   // consumer threads
    static constexpr int A_FLOATS = BM * BK, B_FLOATS = BN * BK;
    static constexpr int STAGE_FLOATS = A_FLOATS + B_FLOATS;
    static constexpr int STAGE_BYTES = STAGE_FLOATS * 4;
    // ring + 1 KiB for aligning the base to the 1 KiB swizzle atom + full and
    // empty barriers
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 16 * STAGES;
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
// moving right, so the CTAs resident together share A row-panels and B
// column-panels in L2 (GROUP * BM = 1024 rows).  DRAM bytes read by one
// 8192^3 launch (64 x 128 tiles, 304 resident CTAs): 5.41 GB for groups of
// 512 rows, 3.79 GB for 1024, 4.74 GB for 2048, 7.95 GB for 4096; the time is
// the same for all four (the FP32 pipe is the bound).
template <int BM>
__device__ __forceinline__ void tile_coords(int bid, int tiles_m, int tiles_n, int &tm, int &tn) {
    constexpr int GROUP = BM >= 1024 ? 1 : 1024 / BM;
    const long long per_group = (long long)GROUP * tiles_n;
    const int g = int(bid / per_group);
    const int first_m = g * GROUP;
    const int gm = min(tiles_m - first_m, GROUP);
    const int in_group = int(bid - g * per_group);
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

// Packed FP32 adds (pack2, add2_rn, fold2): packed_f32.cuh.

// A thread's accumulators, held in pairs: along n when A is K-inner, along m
// when A is MN-inner (the two products of a pair are independent scalars).
template <class T, bool A_KIN>
struct PackedAcc {
    static constexpr bool PAIR_N = A_KIN;
    static constexpr int R = PAIR_N ? T::TM : T::TM / 2;
    static constexpr int C = PAIR_N ? T::TN / 2 : T::TN;
    u64 v[R][C];

    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int j = 0; j < C; ++j) v[i][j] = 0ull;   // two +0.0f
    }

    __device__ __forceinline__ void to_float(float (&f)[T::TM][T::TN]) const {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int j = 0; j < C; ++j) {
                float lo, hi;
                unpack2(v[i][j], lo, hi);
                if (PAIR_N) { f[i][2 * j] = lo; f[i][2 * j + 1] = hi; }
                else        { f[2 * i][j] = lo; f[2 * i + 1][j] = hi; }
            }
    }
};

// One stage (32 k-steps) of the serial k-chain for this thread's accumulators.
// k advances in increasing order: k4 (chunks of 4), then kk.
template <class T, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void mma_stage(const float *__restrict__ As, const float *__restrict__ Bs,
                                          int abase, int bbase, int lm, int ln,
                                          PackedAcc<T, A_KIN> &acc) {
#pragma unroll(K4Unroll<A_KIN, B_KIN>::value)
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
            if constexpr (PackedAcc<T, A_KIN>::PAIR_N) {
                // column pairs outer: measured 0.7% faster at 8192^3 than rows outer
#pragma unroll
                for (int j = 0; j < T::TN / 2; ++j)
#pragma unroll
                    for (int r = 0; r < T::TM; ++r)
                        acc.v[r][j] = fold2(acc.v[r][j], a[r][kk], b[2 * j][kk], a[r][kk], b[2 * j + 1][kk]);
            } else {
#pragma unroll
                for (int i = 0; i < T::TM / 2; ++i)
#pragma unroll
                    for (int c = 0; c < T::TN; ++c)
                        acc.v[i][c] = fold2(acc.v[i][c], a[2 * i][kk], b[c][kk], a[2 * i + 1][kk], b[c][kk]);
            }
        }
    }
}

// Batch strides and epilogue of the EX kernels (kernel parameter).
struct ExArgs {
    int64_t sA, sB, sC;    // batch strides of the operands, elements (cp.async path)
    int zA, zB;            // TMA: 1 when the operand's map has a batch dimension
    float alpha;
    const float *bias;     // N values or null
    int act;               // 0 none, 1 GeLU
    const float *R;        // residual of batch 0 or null; batch b at R + b*sR
    int64_t ldr, sR;
    int64_t causal;        // >= 0: a tile wholly above j = causal + i is skipped
    int64_t k_lo, k_hi;    // >= 0: row i's k-chain covers [i - k_lo, i + k_hi] only
    int b_group;           // batch b reads B_(b / b_group)
    DbgSpan da, db, dc;    // checked build: the spans of A, B and C,
    DbgSpan dsk;           // of the chained split's scratch,
    unsigned *dstat;       // and the status word
};

// Writes the thread's results; rows/columns past M/N are skipped.
template <class T, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void store_acc(float *__restrict__ C, int64_t ldc, int64_t M, int64_t N,
                                          int64_t m0, int64_t n0, int abase, int bbase,
                                          const float (&acc)[T::TM][T::TN], bool c_vec, const ExArgs &ep) {
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
                    if (REPOPS_DBG_OK(ep.dc, crow + gn, 16, ep.dstat))
                        *reinterpret_cast<float4 *>(crow + gn) =
                            make_float4(acc[r][4 * q], acc[r][4 * q + 1], acc[r][4 * q + 2], acc[r][4 * q + 3]);
                } else {
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (gn + t < N && REPOPS_DBG_OK(ep.dc, crow + gn + t, 4, ep.dstat))
                            crow[gn + t] = acc[r][4 * q + t];
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < T::TN; ++c) {
                const int64_t gn = n0 + b_col<true>(bbase, c);
                if (gn < N && REPOPS_DBG_OK(ep.dc, crow + gn, 4, ep.dstat)) crow[gn] = acc[r][c];
            }
        }
    }
}

template <class T, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void store_tile(float *__restrict__ C, int64_t ldc, int64_t M, int64_t N,
                                           int64_t m0, int64_t n0, int abase, int bbase,
                                           const PackedAcc<T, A_KIN> &pacc, bool c_vec, const ExArgs &ep) {
    float acc[T::TM][T::TN];
    pacc.to_float(acc);
    store_acc<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec, ep);
}


// True when every element (i, j) of the tile has j > causal + i: the tile is
// neither computed nor written.
template <int BM>
__device__ __forceinline__ bool tile_above_causal(const ExArgs &ep, int64_t m0, int64_t n0) {
    return ep.causal >= 0 && n0 > m0 + (BM - 1) + ep.causal;
}

// The k-slices [kb, ke) a tile of rows m0 .. m0+BM-1 runs: the union of its
// rows' k windows, widened to whole slices (all KT slices without a band).
// Terms outside a row's own window multiply A entries that the caller keeps
// at +-0 by finite B values: they add +-0 and change no bit.
template <int BM>
__device__ __forceinline__ void tile_k_range(const ExArgs &ep, int64_t m0, int64_t K, int &kb, int &ke) {
    int64_t lo = 0, hi = K;                                   // k in [lo, hi)
    if (ep.k_lo >= 0 && m0 - ep.k_lo > 0) lo = m0 - ep.k_lo;
    if (ep.k_hi >= 0 && m0 + (BM - 1) + ep.k_hi + 1 < hi) hi = m0 + (BM - 1) + ep.k_hi + 1;
    kb = int(lo / BK);
    ke = lo < hi ? int((hi + BK - 1) / BK) : kb;
}

// The epilogue after the whole k-chain of every element, then the store.
// Unrolled over the thread's TM x TN results (registers, independent chains);
// fl(1 * acc) = acc, so alpha = 1 skips the multiply.
template <class T, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void store_tile_ex(float *__restrict__ C, int64_t ldc, int64_t M, int64_t N,
                                              int64_t m0, int64_t n0, int abase, int bbase,
                                              const PackedAcc<T, A_KIN> &pacc, bool c_vec, const ExArgs &ep,
                                              const float *__restrict__ Rb) {
    float acc[T::TM][T::TN];
    pacc.to_float(acc);
    if (ep.alpha != 1.0f) {
#pragma unroll
        for (int r = 0; r < T::TM; ++r)
#pragma unroll
            for (int c = 0; c < T::TN; ++c) acc[r][c] = __fmul_rn(acc[r][c], ep.alpha);
    }
    if (ep.bias) {
#pragma unroll
        for (int c = 0; c < T::TN; ++c) {
            const int64_t gn = n0 + b_col<B_KIN>(bbase, c);
            const float bv = gn < N ? ep.bias[gn] : 0.0f;   // columns past N are not stored
#pragma unroll
            for (int r = 0; r < T::TM; ++r) acc[r][c] = __fadd_rn(acc[r][c], bv);
        }
    }
    if (ep.act == 1) {
        // four independent GeLUs per trip of a loop that is not unrolled:
        // the fully unrolled form (TM*TN inlined copies) measured slower, its
        // code crowding out the main loop of the CTA sharing the SM
        float v[T::TM * T::TN];
#pragma unroll
        for (int r = 0; r < T::TM; ++r)
#pragma unroll
            for (int c = 0; c < T::TN; ++c) v[r * T::TN + c] = acc[r][c];
#pragma unroll 1
        for (int e = 0; e < T::TM * T::TN; e += 4) {
            const float y0 = gelu_fixed(v[e]), y1 = gelu_fixed(v[e + 1]);
            const float y2 = gelu_fixed(v[e + 2]), y3 = gelu_fixed(v[e + 3]);
            v[e] = y0; v[e + 1] = y1; v[e + 2] = y2; v[e + 3] = y3;
        }
#pragma unroll
        for (int r = 0; r < T::TM; ++r)
#pragma unroll
            for (int c = 0; c < T::TN; ++c) acc[r][c] = v[r * T::TN + c];
    }
    if (Rb) {
#pragma unroll
        for (int r = 0; r < T::TM; ++r) {
            const int64_t gm = m0 + a_row<A_KIN>(abase, r);
            if (gm >= M) break;   // rows increase with r; later rows are not stored
#pragma unroll
            for (int c = 0; c < T::TN; ++c) {
                const int64_t gn = n0 + b_col<B_KIN>(bbase, c);
                if (gn < N) acc[r][c] = __fadd_rn(acc[r][c], Rb[gm * ep.ldr + gn]);
            }
        }
    }
    store_acc<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec, ep);
}

__device__ __forceinline__ float *aligned_smem_base(unsigned char *raw) {
    return reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------------ TMA ----

// THREADS consumer threads plus one producer warp.  The producer's lane 0
// refills ring slot s with TMA once every consumer warp has arrived on
// empty[s]; consumers wait on full[s] (TMA transaction bytes) and never
// synchronise the whole CTA, so warps drift within the ring instead of meeting
// at a barrier every k-slice.  Every wait is bounded; on a timeout the status
// bit is set, the producer lets its in-flight copies land, and the tile is not
// stored.
template <class T, bool A_KIN, bool B_KIN, bool EX>
__global__ void __launch_bounds__(T::THREADS + 32, T::MINB)
gemm_tma_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   float *__restrict__ C, int64_t M, int64_t N, int64_t K, int64_t ldc,
                   int tiles_m, int tiles_n, int c_vec, unsigned *status, const ExArgs ep) {
    constexpr int CONSUMER_WARPS = T::THREADS / 32;
    extern __shared__ unsigned char smem_raw[];
    float *smem = aligned_smem_base(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + T::STAGES * T::STAGE_FLOATS);
    uint64_t *empty = full + T::STAGES;

    const int tid = threadIdx.x;
    int tm, tn;
    tile_coords<T::BM>(blockIdx.x, tiles_m, tiles_n, tm, tn);
    if (EX && ep.k_hi >= 0) tm = tiles_m - 1 - tm;             // longest k-ranges first
    const int64_t m0 = int64_t(tm) * T::BM, n0 = int64_t(tn) * T::BN;
    int kb = 0, ke = int((K + BK - 1) / BK);
    if constexpr (EX) tile_k_range<T::BM>(ep, m0, K, kb, ke);
    const int NKT = ke - kb;                                   // slices this tile runs
    if (EX && tile_above_causal<T::BM>(ep, m0, n0)) return;   // the whole CTA, before any barrier

    if (tid == T::THREADS) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
#pragma unroll 1
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CONSUMER_WARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= T::THREADS) {   // producer warp
        if (tid == T::THREADS) {
            int issued = 0;
            bool ok = true;
#pragma unroll 1
            for (int kt = 0; kt < NKT; ++kt) {
                const int s = kt % T::STAGES;
                if (kt >= T::STAGES &&
                    !mbar_wait_bounded(&empty[s], uint32_t(kt / T::STAGES - 1) & 1u)) {
                    ok = false;
                    break;
                }
                float *As = smem + s * T::STAGE_FLOATS;
                float *Bs = As + T::A_FLOATS;
                mbar_arrive_expect_tx(&full[s], T::STAGE_BYTES);
                const int k0 = (kb + kt) * BK;
                const int ax = A_KIN ? k0 : int(m0), ay = A_KIN ? int(m0) : k0;
                const int bx = B_KIN ? k0 : int(n0), by = B_KIN ? int(n0) : k0;
                if (EX && ep.zA) tma_load_3d(As, &tmA, &full[s], ax, ay, int(blockIdx.y));
                else             tma_load_2d(As, &tmA, &full[s], ax, ay);
                if (EX && ep.zB) tma_load_3d(Bs, &tmB, &full[s], bx, by, int(blockIdx.y) / ep.b_group);
                else             tma_load_2d(Bs, &tmB, &full[s], bx, by);
                issued = kt + 1;
            }
            if (!ok) atomicOr(status, 1u);
            // every copy in flight must land before the CTA's shared memory is released
#pragma unroll 1
            for (int kt = max(0, issued - T::STAGES); kt < issued; ++kt)
                mbar_wait_bounded(&full[kt % T::STAGES], uint32_t(kt / T::STAGES) & 1u);
        }
        return;
    }

    const int warp = tid >> 5, lane = tid & 31;
    const int warp_m = warp % T::WARPS_M, warp_n = warp / T::WARPS_M;
    const int lm = lane >> 3, ln = lane & 7;
    const int abase = warp_m * T::WM + (A_KIN ? lm : lm * T::TM);
    const int bbase = warp_n * T::WN + (B_KIN ? ln : ln * 4);

    PackedAcc<T, A_KIN> acc;
    acc.zero();
#pragma unroll 1
    for (int kt = 0; kt < NKT; ++kt) {
        const int s = kt % T::STAGES;
        if (!mbar_wait_bounded(&full[s], uint32_t(kt / T::STAGES) & 1u)) {
            atomicOr(status, 1u);
            return;
        }
        const float *As = smem + s * T::STAGE_FLOATS;
        mma_stage<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, abase, bbase, lm, ln, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if constexpr (EX) {
        const int64_t b = blockIdx.y;
        store_tile_ex<T, A_KIN, B_KIN>(C + b * ep.sC, ldc, M, N, m0, n0, abase, bbase, acc, c_vec != 0, ep,
                                       ep.R ? ep.R + b * ep.sR : nullptr);
    } else {
        store_tile<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec != 0, ep);
    }
}

// ------------------------------------------------------- chained k-split ----
//
// The same warp-specialised TMA pipeline run by a persistent grid of `workers`
// CTAs that together balance the work when the tile count is not a multiple of
// the resident CTAs.  Whole waves first: worker w runs tiles i*workers + w,
// exactly as the one-tile-per-CTA kernel's resident CTAs would.  The remaining
// tiles (more than `workers`, fewer than twice as many) are cut into k-slices,
// and worker w takes an equal share of those slices in tile order, so a tile
// may be split between two consecutive workers.  A split tile's k-chains are
// CONTINUED, never reordered: worker w-1 runs slices [0, h) of the tile from
// +0 and stores every accumulator as it stands (a binary32 value, stored and
// loaded exactly); worker w loads them and runs slices [h, KT), so every
// element still sees k = 0, 1, 2, ... in one serial chain of separately
// rounded products and sums -- the same operations, the same bits.
//
// Worker w runs its share's head (the first part of its last tile) before the
// tail (the rest of its first tile), so the head worker w-1 stores is ready
// long before w needs it: w reaches its tail after (share - (KT - h)) >= h
// slices of its own split work.  Every wait is bounded.  The grid is launched
// cooperatively (all workers resident), which the waits between workers need.
struct SkArgs {
    int64_t dp_tiles;    // tiles run whole, one per worker per wave (waves * workers)
    int64_t sk_tiles;    // the remaining tiles, split by k-slices
    int kt;              // k-slices of a whole tile
    int waves;
    u64 *partial;        // [workers][pairs per thread][THREADS] accumulator pairs
    unsigned *flags;     // [workers][THREADS], zero before the launch
};

// The schedule of `tiles` tiles of kt k-slices over `workers` workers
// (workers <= tiles): whole waves while more than one wave of tiles is left,
// then the rest split by k-slices.  Host and device agree on it through
// SkPlan below; a host test checks its invariants.
inline void sk_schedule(int64_t tiles, int kt, int workers, SkArgs &sk) {
    sk.kt = kt;
    if (tiles % workers == 0) {
        sk.waves = int(tiles / workers);
        sk.sk_tiles = 0;
    } else {
        sk.waves = int(tiles / workers) - 1;
        sk.sk_tiles = tiles - int64_t(sk.waves) * workers;
    }
    sk.dp_tiles = int64_t(sk.waves) * workers;
}

// One piece of a worker's schedule.  kind 0: slices [kb, ke) from +0, then
// store the accumulators for the next worker (a head); 1: a whole tile; 2:
// load the previous worker's accumulators, slices [kb, ke), store C (a tail).
struct SkSeg {
    int64_t tile;
    int kb, ke, kind;
};

struct SkPlan {
    int waves, w;
    int64_t dp_tiles, workers;
    int kt;
    int64_t t_first, t_last;   // split tiles touched (absolute tile indices)
    int k_first, k_end;        // the share starts at slice k_first of t_first, ends before k_end of t_last
    int has_head, has_tail;
    int64_t full_first, nfull;
    int nseg;

    __host__ __device__ __forceinline__ SkPlan(const SkArgs &sk, int w_, int workers_) {
        waves = sk.waves;
        w = w_;
        workers = workers_;
        dp_tiles = sk.dp_tiles;
        kt = sk.kt;
        has_head = has_tail = 0;
        nfull = 0;
        full_first = 0;
        t_first = t_last = 0;
        k_first = 0;
        k_end = kt;
        if (sk.sk_tiles > 0) {
            const int64_t units = sk.sk_tiles * kt;
            const int64_t q = units / workers, r = units % workers;
            const int64_t u0 = q * w + (w < r ? w : r);
            const int64_t u1 = u0 + q + (w < r ? 1 : 0);
            t_first = dp_tiles + u0 / kt;
            k_first = int(u0 % kt);
            t_last = dp_tiles + (u1 - 1) / kt;
            k_end = int((u1 - 1) % kt) + 1;
            has_head = k_end < kt;
            has_tail = k_first > 0;
            full_first = t_first + has_tail;
            nfull = (t_last - has_head) - full_first + 1;
            if (nfull < 0) nfull = 0;
        }
        nseg = waves + has_head + int(nfull) + has_tail;
    }

    // Segment s in execution order: whole waves, the head, whole split-part
    // tiles, the tail.
    __host__ __device__ __forceinline__ SkSeg seg(int s) const {
        SkSeg g;
        if (s < waves) {
            g.tile = int64_t(s) * workers + w; g.kb = 0; g.ke = kt; g.kind = 1;
            return g;
        }
        s -= waves;
        if (has_head) {
            if (s == 0) { g.tile = t_last; g.kb = 0; g.ke = k_end; g.kind = 0; return g; }
            --s;
        }
        if (s < nfull) {
            g.tile = full_first + s; g.kb = 0; g.ke = kt; g.kind = 1;
            return g;
        }
        g.tile = t_first; g.kb = k_first; g.ke = kt; g.kind = 2;
        return g;
    }
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits until *flag is non-zero; gives up after limit_ns.
__device__ __forceinline__ bool flag_wait_bounded_ns(const unsigned *flag, uint64_t limit_ns) {
    if (ld_acquire_gpu(flag)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i) {
            __nanosleep(64);
            if (ld_acquire_gpu(flag)) return true;
        }
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// Waits until *flag is non-zero; gives up after kWaitLimitNs.
__device__ __forceinline__ bool flag_wait_bounded(const unsigned *flag) {
    return flag_wait_bounded_ns(flag, kWaitLimitNs);
}

template <class T, bool A_KIN, bool B_KIN, bool EX>
__global__ void __launch_bounds__(T::THREADS + 32, T::MINB)
gemm_tma_sk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   float *__restrict__ C, int64_t M, int64_t N, int64_t K, int64_t ldc,
                   int tiles_m, int tiles_n, int c_vec, unsigned *status, const ExArgs ep, const SkArgs sk) {
    constexpr int CONSUMER_WARPS = T::THREADS / 32;
    constexpr int PAIRS = PackedAcc<T, A_KIN>::R * PackedAcc<T, A_KIN>::C;
    extern __shared__ unsigned char smem_raw[];
    float *smem = aligned_smem_base(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + T::STAGES * T::STAGE_FLOATS);
    uint64_t *empty = full + T::STAGES;

    const int tid = threadIdx.x;
    const SkPlan plan(sk, int(blockIdx.x), int(gridDim.x));

    if (tid == T::THREADS) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
#pragma unroll 1
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CONSUMER_WARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= T::THREADS) {   // producer warp: every slice of every segment, in order
        if (tid == T::THREADS) {
            int issued = 0;
            bool ok = true;
#pragma unroll 1
            for (int si = 0; si < plan.nseg && ok; ++si) {
                const SkSeg g = plan.seg(si);
                int tm, tn;
                tile_coords<T::BM>(int(g.tile), tiles_m, tiles_n, tm, tn);
                const int m0 = tm * T::BM, n0 = tn * T::BN;
#pragma unroll 1
                for (int k = g.kb; k < g.ke; ++k) {
                    const int s = issued % T::STAGES;
                    if (issued >= T::STAGES &&
                        !mbar_wait_bounded(&empty[s], uint32_t(issued / T::STAGES - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    float *As = smem + s * T::STAGE_FLOATS;
                    float *Bs = As + T::A_FLOATS;
                    mbar_arrive_expect_tx(&full[s], T::STAGE_BYTES);
                    const int k0 = k * BK;
                    tma_load_2d(As, &tmA, &full[s], A_KIN ? k0 : m0, A_KIN ? m0 : k0);
                    tma_load_2d(Bs, &tmB, &full[s], B_KIN ? k0 : n0, B_KIN ? n0 : k0);
                    ++issued;
                }
            }
            if (!ok) atomicOr(status, 1u);
#pragma unroll 1
            for (int it = max(0, issued - T::STAGES); it < issued; ++it)
                mbar_wait_bounded(&full[it % T::STAGES], uint32_t(it / T::STAGES) & 1u);
        }
        return;
    }

    const int warp = tid >> 5, lane = tid & 31;
    const int warp_m = warp % T::WARPS_M, warp_n = warp / T::WARPS_M;
    const int lm = lane >> 3, ln = lane & 7;
    const int abase = warp_m * T::WM + (A_KIN ? lm : lm * T::TM);
    const int bbase = warp_n * T::WN + (B_KIN ? ln : ln * 4);
    const int64_t w = blockIdx.x;

    int consumed = 0;
#pragma unroll 1
    for (int si = 0; si < plan.nseg; ++si) {
        const SkSeg g = plan.seg(si);
        int tm, tn;
        tile_coords<T::BM>(int(g.tile), tiles_m, tiles_n, tm, tn);
        const int64_t m0 = int64_t(tm) * T::BM, n0 = int64_t(tn) * T::BN;
        PackedAcc<T, A_KIN> acc;
        if (g.kind == 2) {
            // continue the chains the previous worker stored (its head of this tile)
            if (!REPOPS_DBG_OK(ep.dsk, sk.flags + (w - 1) * T::THREADS + tid, 4, ep.dstat) ||
                !flag_wait_bounded(sk.flags + (w - 1) * T::THREADS + tid)) {
                atomicOr(status, 1u);
                return;
            }
            const u64 *src = sk.partial + (w - 1) * int64_t(PAIRS) * T::THREADS + tid;
#pragma unroll
            for (int i = 0; i < PackedAcc<T, A_KIN>::R; ++i)
#pragma unroll
                for (int j = 0; j < PackedAcc<T, A_KIN>::C; ++j)
                    acc.v[i][j] = REPOPS_DBG_OK(ep.dsk, src + (i * PackedAcc<T, A_KIN>::C + j) * T::THREADS, 8,
                                                ep.dstat)
                                      ? __ldcg(src + (i * PackedAcc<T, A_KIN>::C + j) * T::THREADS)
                                      : 0ull;
        } else {
            acc.zero();
        }
#pragma unroll 1
        for (int k = g.kb; k < g.ke; ++k) {
            const int s = consumed % T::STAGES;
            if (!mbar_wait_bounded(&full[s], uint32_t(consumed / T::STAGES) & 1u)) {
                atomicOr(status, 1u);
                return;
            }
            const float *As = smem + s * T::STAGE_FLOATS;
            mma_stage<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, abase, bbase, lm, ln, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++consumed;
        }
        if (g.kind == 0) {
            // the accumulators as they stand, for worker w + 1 (same thread index,
            // same element mapping); then release them
            u64 *dst = sk.partial + w * int64_t(PAIRS) * T::THREADS + tid;
#pragma unroll
            for (int i = 0; i < PackedAcc<T, A_KIN>::R; ++i)
#pragma unroll
                for (int j = 0; j < PackedAcc<T, A_KIN>::C; ++j)
                    if (REPOPS_DBG_OK(ep.dsk, dst + (i * PackedAcc<T, A_KIN>::C + j) * T::THREADS, 8, ep.dstat))
                        dst[(i * PackedAcc<T, A_KIN>::C + j) * T::THREADS] = acc.v[i][j];
            if (REPOPS_DBG_OK(ep.dsk, sk.flags + w * T::THREADS + tid, 4, ep.dstat))
                st_release_gpu(sk.flags + w * T::THREADS + tid, 1u);
        } else if constexpr (EX) {
            store_tile_ex<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec != 0, ep, ep.R);
        } else {
            store_tile<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec != 0, ep);
        }
    }
}

// ------------------------------------------------------------- cp.async ----

// Fills one ring slot with k-slice [k0, k0 + 32) of both operands, 4 bytes per
// copy, zero-filling everything outside the matrices.
template <class T, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void load_slice_cpasync(float *As, float *Bs, const float *__restrict__ A,
                                                   int64_t lda, const float *__restrict__ B, int64_t ldb,
                                                   int64_t M, int64_t N, int64_t K,
                                                   int64_t m0, int64_t n0, int64_t k0, int tid, const ExArgs &ep) {
    constexpr int NW = T::THREADS / 32;
    if constexpr (A_KIN) {
        // element (r, k): a warp copies one 128-byte row segment
        const int k = tid & 31;
        const int64_t gk = k0 + k;
#pragma unroll 4
        for (int r = tid >> 5; r < T::BM; r += NW) {
            const int64_t gm = m0 + r;
            const bool ok = gk < K && gm < M && REPOPS_DBG_OK(ep.da, A + gm * lda + gk, 4, ep.dstat);
            cp_async_4(As + kin_off(r, k), ok ? A + gm * lda + gk : A, ok ? 4u : 0u);
        }
    } else {
#pragma unroll 4
        for (int e = tid; e < BK * T::BM; e += T::THREADS) {
            const int k = e / T::BM, r = e % T::BM;
            const int64_t gk = k0 + k, gm = m0 + r;
            const bool ok = gk < K && gm < M && REPOPS_DBG_OK(ep.da, A + gk * lda + gm, 4, ep.dstat);
            cp_async_4(As + k * T::BM + r, ok ? A + gk * lda + gm : A, ok ? 4u : 0u);
        }
    }
    if constexpr (B_KIN) {
        const int k = tid & 31;
        const int64_t gk = k0 + k;
#pragma unroll 4
        for (int r = tid >> 5; r < T::BN; r += NW) {
            const int64_t gn = n0 + r;
            const bool ok = gk < K && gn < N && REPOPS_DBG_OK(ep.db, B + gn * ldb + gk, 4, ep.dstat);
            cp_async_4(Bs + kin_off(r, k), ok ? B + gn * ldb + gk : B, ok ? 4u : 0u);
        }
    } else {
#pragma unroll 4
        for (int e = tid; e < BK * T::BN; e += T::THREADS) {
            const int k = e / T::BN, r = e % T::BN;
            const int64_t gk = k0 + k, gn = n0 + r;
            const bool ok = gk < K && gn < N && REPOPS_DBG_OK(ep.db, B + gk * ldb + gn, 4, ep.dstat);
            cp_async_4(Bs + k * T::BN + r, ok ? B + gk * ldb + gn : B, ok ? 4u : 0u);
        }
    }
}

template <class T, bool A_KIN, bool B_KIN, bool EX>
__global__ void __launch_bounds__(T::THREADS, T::MINB)
gemm_cpasync_kernel(const float *__restrict__ A, int64_t lda, const float *__restrict__ B, int64_t ldb,
                    float *__restrict__ C, int64_t M, int64_t N, int64_t K, int64_t ldc,
                    int tiles_m, int tiles_n, int c_vec, const ExArgs ep) {
    extern __shared__ unsigned char smem_raw[];
    float *smem = aligned_smem_base(smem_raw);
    if constexpr (EX) {
        const int64_t b = blockIdx.y;
        A += b * ep.sA;
        B += (b / ep.b_group) * ep.sB;
        C += b * ep.sC;
    }

    const int tid = threadIdx.x;
    int tm, tn;
    tile_coords<T::BM>(blockIdx.x, tiles_m, tiles_n, tm, tn);
    if (EX && ep.k_hi >= 0) tm = tiles_m - 1 - tm;             // longest k-ranges first
    const int64_t m0 = int64_t(tm) * T::BM, n0 = int64_t(tn) * T::BN;
    int kb = 0, ke = int((K + BK - 1) / BK);
    if constexpr (EX) tile_k_range<T::BM>(ep, m0, K, kb, ke);
    const int KT = ke - kb;                                    // slices this tile runs
    if (EX && tile_above_causal<T::BM>(ep, m0, n0)) return;   // the whole CTA, before any barrier

#pragma unroll 1
    for (int s = 0; s < T::STAGES - 1; ++s) {
        if (s < KT) {
            float *As = smem + s * T::STAGE_FLOATS;
            load_slice_cpasync<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, A, lda, B, ldb, M, N, K,
                                                m0, n0, int64_t(kb + s) * BK, tid, ep);
        }
        cp_async_commit();
    }

    const int warp = tid >> 5, lane = tid & 31;
    const int warp_m = warp % T::WARPS_M, warp_n = warp / T::WARPS_M;
    const int lm = lane >> 3, ln = lane & 7;
    const int abase = warp_m * T::WM + (A_KIN ? lm : lm * T::TM);
    const int bbase = warp_n * T::WN + (B_KIN ? ln : ln * 4);

    PackedAcc<T, A_KIN> acc;
    acc.zero();
#pragma unroll 1
    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<T::STAGES - 2>();   // slice kt has landed (this thread's copies)
        __syncthreads();                  // ... and everyone's; slot kt-1 is free
        const int nk = kt + T::STAGES - 1;
        if (nk < KT) {
            float *As = smem + (nk % T::STAGES) * T::STAGE_FLOATS;
            load_slice_cpasync<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, A, lda, B, ldb, M, N, K,
                                                m0, n0, int64_t(kb + nk) * BK, tid, ep);
        }
        cp_async_commit();
        const float *As = smem + (kt % T::STAGES) * T::STAGE_FLOATS;
        mma_stage<T, A_KIN, B_KIN>(As, As + T::A_FLOATS, abase, bbase, lm, ln, acc);
    }
    cp_async_wait<0>();
    if constexpr (EX)
        store_tile_ex<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec != 0, ep,
                                       ep.R ? ep.R + int64_t(blockIdx.y) * ep.sR : nullptr);
    else
        store_tile<T, A_KIN, B_KIN>(C, ldc, M, N, m0, n0, abase, bbase, acc, c_vec != 0, ep);
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

// 3-D fp32 tensor map: as make_map plus a batch dimension of `batch`
// matrices `stride` elements apart (box extent 1 in it).
inline bool make_map_3d(CUtensorMap *map, const float *base, int64_t inner, int64_t outer, int64_t batch,
                        int64_t ld, int64_t stride, int box_inner, int box_outer, bool swizzle128) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {cuuint64_t(inner), cuuint64_t(outer), cuuint64_t(batch)};
    cuuint64_t strides[2] = {cuuint64_t(ld) * 4u, cuuint64_t(stride) * 4u};
    cuuint32_t box[3] = {cuuint32_t(box_inner), cuuint32_t(box_outer), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// An operand's map: 3-D when it advances with the batch (z = 1), else 2-D.
inline bool make_operand_map(CUtensorMap *map, const float *base, int64_t inner, int64_t outer, int64_t ld,
                             int64_t batch, int64_t stride, int z, int box_inner, int box_outer, bool swz) {
    return z ? make_map_3d(map, base, inner, outer, batch, ld, stride, box_inner, box_outer, swz)
             : make_map(map, base, inner, outer, ld, box_inner, box_outer, swz);
}

// The number of distinct B matrices a batched call reads.
inline int64_t b_batches(const GemmProblem &p) { return (p.batch + p.b_group - 1) / p.b_group; }

inline ExArgs ex_args(const GemmProblem &p) {
    ExArgs ep{};
    ep.alpha = 1.0f;
    ep.causal = -1;
    ep.k_lo = ep.k_hi = -1;
    ep.b_group = 1;
    ep.da.lo = p.span_a[0]; ep.da.hi = p.span_a[1];
    ep.db.lo = p.span_b[0]; ep.db.hi = p.span_b[1];
    ep.dc.lo = p.span_c[0]; ep.dc.hi = p.span_c[1];
    ep.dstat = p.status;
    if (!p.ex) return ep;
    ep.sA = p.strideA; ep.sB = p.strideB; ep.sC = p.strideC;
    ep.zA = p.batch > 1 && p.strideA != 0;
    ep.zB = b_batches(p) > 1 && p.strideB != 0;
    ep.alpha = p.alpha;
    ep.bias = p.bias;
    ep.act = p.act;
    ep.R = p.R;
    ep.ldr = p.ldr;
    ep.sR = p.strideR;
    ep.causal = p.causal;
    ep.k_lo = p.k_lo;
    ep.k_hi = p.k_hi;
    ep.b_group = int(p.b_group);
    return ep;
}

template <class T, bool A_KIN, bool B_KIN, bool EX>
int launch_tma(const GemmProblem &p, int tiles_m, int tiles_n, int c_vec) {
    CUtensorMap ma, mb;
    const ExArgs ep = ex_args(p);
    // A: row-major (K-inner) -> dims {K, M}; transposed (M-inner) -> {M, K}
    const bool okA = A_KIN ? make_operand_map(&ma, p.A, p.K, p.M, p.lda, p.batch, p.strideA, ep.zA, BK, T::BM, true)
                           : make_operand_map(&ma, p.A, p.M, p.K, p.lda, p.batch, p.strideA, ep.zA, T::BM, BK, false);
    // B: transposed (K-inner) -> dims {K, N}; row-major (N-inner) -> {N, K}
    const bool okB = B_KIN ? make_operand_map(&mb, p.B, p.K, p.N, p.ldb, b_batches(p), p.strideB, ep.zB, BK, T::BN, true)
                           : make_operand_map(&mb, p.B, p.N, p.K, p.ldb, b_batches(p), p.strideB, ep.zB, T::BN, BK, false);
    if (!okA || !okB) return REPOPS_ERR_UNSUPPORTED;
    auto kern = gemm_tma_ws_kernel<T, A_KIN, B_KIN, EX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return set_cuda_error(e);
    const dim3 grid(unsigned(tiles_m * tiles_n), EX ? unsigned(p.batch) : 1u);
    kern<<<grid, T::THREADS + 32, T::SMEM_BYTES, p.stream>>>(ma, mb, p.C, p.M, p.N, p.K, p.ldc, tiles_m, tiles_n,
                                                             c_vec, p.status, ep);
    return check_launch();
}

// Scratch of the chained k-split: accumulator pairs of every worker's head,
// then one flag per worker thread (zeroed by the caller before each launch).
template <class T>
constexpr size_t sk_partial_bytes(int workers) {
    return size_t(workers) * size_t(T::THREADS) * size_t(T::TM * T::TN) * 4u;
}

template <class T, bool A_KIN, bool B_KIN, bool EX>
int launch_tma_sk(const GemmProblem &p, int tiles_m, int tiles_n, int c_vec) {
    if (p.batch != 1 || (p.ex && (p.causal >= 0 || p.k_lo >= 0 || p.k_hi >= 0))) return REPOPS_ERR_UNSUPPORTED;
    CUtensorMap ma, mb;
    const ExArgs ep = ex_args(p);
    const bool okA = A_KIN ? make_map(&ma, p.A, p.K, p.M, p.lda, BK, T::BM, true)
                           : make_map(&ma, p.A, p.M, p.K, p.lda, T::BM, BK, false);
    const bool okB = B_KIN ? make_map(&mb, p.B, p.K, p.N, p.ldb, BK, T::BN, true)
                           : make_map(&mb, p.B, p.N, p.K, p.ldb, T::BN, BK, false);
    if (!okA || !okB) return REPOPS_ERR_UNSUPPORTED;
    auto kern = gemm_tma_sk_kernel<T, A_KIN, B_KIN, EX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return set_cuda_error(e);
    // every worker must be resident at once (the cooperative launch checks it too)
    int per_sm = 0, dev = 0, sms = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, T::THREADS + 32, T::SMEM_BYTES)) !=
            cudaSuccess ||
        (e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return set_cuda_error(e);
    const int64_t tiles = int64_t(tiles_m) * tiles_n;
    const int workers = p.sk_workers;
    if (workers < 1 || workers > int64_t(per_sm) * sms || workers > tiles) return REPOPS_ERR_UNSUPPORTED;
    SkArgs sk{};
    sk_schedule(tiles, int((p.K + BK - 1) / BK), workers, sk);
    sk.partial = static_cast<u64 *>(p.sk_scratch);
    sk.flags = reinterpret_cast<unsigned *>(static_cast<unsigned char *>(p.sk_scratch) +
                                            sk_partial_bytes<T>(workers));
    ExArgs eps = ep;
    eps.dsk = dbg_span(p.sk_scratch, sk_partial_bytes<T>(workers) + size_t(workers) * T::THREADS * 4u);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(workers), 1u, 1u);
    cfg.blockDim = dim3(unsigned(T::THREADS + 32), 1u, 1u);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cfg.stream = p.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, ma, mb, p.C, p.M, p.N, p.K, p.ldc, tiles_m, tiles_n, c_vec, p.status, eps,
                           sk);
    if (e != cudaSuccess) return set_cuda_error(e);
    return check_launch();
}

template <class T, bool A_KIN, bool B_KIN, bool EX>
int launch_cpasync(const GemmProblem &p, int tiles_m, int tiles_n, int c_vec) {
    auto kern = gemm_cpasync_kernel<T, A_KIN, B_KIN, EX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return set_cuda_error(e);
    const dim3 grid(unsigned(tiles_m * tiles_n), EX ? unsigned(p.batch) : 1u);
    kern<<<grid, T::THREADS, T::SMEM_BYTES, p.stream>>>(p.A, p.lda, p.B, p.ldb, p.C, p.M, p.N, p.K, p.ldc,
                                                        tiles_m, tiles_n, c_vec, ex_args(p));
    return check_launch();
}

template <class T, bool EX>
int launch_layout(const GemmProblem &p, int loader, int tmi, int tni, int c_vec) {
    const bool a_kin = p.transA == 0, b_kin = p.transB != 0;
    if (loader == REPOPS_LOADER_TMA && p.sk_workers > 0) {
        if (a_kin && !b_kin) return launch_tma_sk<T, true, false, EX>(p, tmi, tni, c_vec);
        if (a_kin && b_kin) return launch_tma_sk<T, true, true, EX>(p, tmi, tni, c_vec);
        if (!a_kin && !b_kin) return launch_tma_sk<T, false, false, EX>(p, tmi, tni, c_vec);
        return launch_tma_sk<T, false, true, EX>(p, tmi, tni, c_vec);
    }
    if (loader == REPOPS_LOADER_TMA) {
        if (a_kin && !b_kin) return launch_tma<T, true, false, EX>(p, tmi, tni, c_vec);
        if (a_kin && b_kin) return launch_tma<T, true, true, EX>(p, tmi, tni, c_vec);
        if (!a_kin && !b_kin) return launch_tma<T, false, false, EX>(p, tmi, tni, c_vec);
        return launch_tma<T, false, true, EX>(p, tmi, tni, c_vec);
    }
    if (a_kin && !b_kin) return launch_cpasync<T, true, false, EX>(p, tmi, tni, c_vec);
    if (a_kin && b_kin) return launch_cpasync<T, true, true, EX>(p, tmi, tni, c_vec);
    if (!a_kin && !b_kin) return launch_cpasync<T, false, false, EX>(p, tmi, tni, c_vec);
    return launch_cpasync<T, false, true, EX>(p, tmi, tni, c_vec);
}

// loader: REPOPS_LOADER_TMA or REPOPS_LOADER_CPASYNC (already resolved).
template <class T>
int launch_config(const GemmProblem &p, int loader) {
    const int64_t tiles_m = (p.M + T::BM - 1) / T::BM;
    const int64_t tiles_n = (p.N + T::BN - 1) / T::BN;
    if (tiles_m * tiles_n > 0x7fffffffLL) return REPOPS_ERR_UNSUPPORTED;
    // C of every batch is 16-byte aligned with a 16-byte pitch
    const int c_vec = (reinterpret_cast<uintptr_t>(p.C) % 16 == 0) && (p.ldc % 4 == 0) &&
                      (!p.ex || p.strideC % 4 == 0);
    const int tmi = int(tiles_m), tni = int(tiles_n);
    return p.ex ? launch_layout<T, true>(p, loader, tmi, tni, c_vec)
                : launch_layout<T, false>(p, loader, tmi, tni, c_vec);
}

// Resident CTAs per SM of the TMA kernel (row-major operands) on the current device.
template <class T>
int occupancy() {
    auto kern = gemm_tma_ws_kernel<T, true, false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, T::THREADS + 32, T::SMEM_BYTES) != cudaSuccess)
        return 0;
    return n;
}

template <class T>
GemmConfigInfo info() {
    return GemmConfigInfo{T::BM, T::BN, T::THREADS, T::TM, T::TN, T::STAGES};
}

// Bytes of chained k-split scratch for `workers` workers: their heads'
// accumulators, then one flag per worker thread (the last workers * THREADS * 4
// bytes, which the caller zeroes before the launch).
template <class T>
size_t sk_scratch_bytes(int workers) {
    return sk_partial_bytes<T>(workers) + size_t(workers) * size_t(T::THREADS) * 4u;
}

}  // namespace gemm
}  // namespace repops

// Defines the three entry points of one configuration.
#define REPOPS_DEFINE_GEMM_CONFIG(N, TILE)                                                        \
    namespace repops {                                                                            \
    int gemm_launch_cfg##N(const GemmProblem &p, int loader) { return gemm::launch_config<TILE>(p, loader); } \
    int gemm_occupancy_cfg##N() { return gemm::occupancy<TILE>(); }                               \
    GemmConfigInfo gemm_info_cfg##N() { return gemm::info<TILE>(); }                              \
    size_t gemm_sk_scratch_cfg##N(int workers) { return gemm::sk_scratch_bytes<TILE>(workers); }  \
    }
