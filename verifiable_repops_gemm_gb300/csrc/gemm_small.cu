// gemm_small.cu -- the order-fixed GEMM for outputs too small to fill the GPU
// with the tiled kernels' CTA tiles (a 256 x 256 output is 32 CTAs of 32 x 64
// on 152 SMs).
//
// "Verde与RepOps" §3.2 (matmul example): each C[i][j] is one k-chain, products
// rounded to binary32 and added in increasing k from +0.  The chains are the
// same as in the tiled kernels -- only the launch shape differs: 16 x 32 CTA
// tiles of 128 threads, each thread two rows by two columns, operands staged
// in k-chunks of 64 through a 3-deep cp.async ring (4-byte copies, any
// alignment, either storage order; 39 KB of shared memory), so a 256^3
// problem runs as 128 CTAs.  Measured on GB300, CUDA-graph replays (operands
// in L2): 256^3 in 4.4 us against 9.5 us on the tiled kernels (6.0 us for the
// library's FP32 GEMM with fused multiply-adds); 384^3 8.4 against 13.1 us;
// 512^3 18.8 against 16.9 us, where the tiled kernels take over.  Computing
// each copy's address once per thread instead of per chunk took 256^3 from
// 9.5 to 5.3 us, chunks of 64 instead of 32 to 4.4 us; one output per thread
// row (8 x 32 tiles, twice the warps) was slower from 256^3 up.
#include "gemm_common.h"
#include "gemm_kernels.cuh"
#include "internal.cuh"
#include "repops.h"

namespace repops {
namespace {

constexpr int kSmBM = 16, kSmBN = 32, kSmKC = 64;   // CTA tile and k-chunk
constexpr int kSmThreads = 128;                      // 8 x 16 threads, 2 x 2 outputs each
constexpr int kSmLdA = kSmBM + 2, kSmLdB = kSmBN + 2;   // padded rows (even: 8-byte reads)

template <int STAGES>
struct SmallSmem {
    float a[STAGES][kSmKC][kSmLdA];   // a[s][k][i] = A[m0 + i][k0 + k]
    float b[STAGES][kSmKC][kSmLdB];   // b[s][k][j] = B[k0 + k][n0 + j]
};

// A thread's share of staging one k-chunk: kRA elements of A and kRB of B.
// Their positions inside the chunk are fixed, so each copy's source offset,
// shared-memory address and row/column test are computed once; chunk c adds
// c * inc to the offsets.  Consecutive threads walk each operand's inner
// (contiguous) index.  Elements past M, N or K are filled with +0 in both
// operands, so a padded step adds fl(0 * 0) = +0 to an accumulator that is
// never -0: the chain is unchanged.
constexpr int kRA = kSmBM * kSmKC / kSmThreads, kRB = kSmBN * kSmKC / kSmThreads;

__device__ __forceinline__ void cp_async_4_to(uint32_t dst, const float *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// The checked build's spans of A, B and C and the status word (unused in the
// release build).
struct SmallDbg {
    DbgSpan a, b, c;
    unsigned *status;
};

template <int STAGES>
__global__ void __launch_bounds__(kSmThreads)
gemm_small_kernel(int transA, int transB, int64_t M, int64_t N, int64_t K,
                  const float *__restrict__ A, int64_t lda, const float *__restrict__ B, int64_t ldb,
                  float *__restrict__ C, int64_t ldc, const SmallDbg dbg) {
    extern __shared__ __align__(16) unsigned char small_smem_raw[];
    SmallSmem<STAGES> &sm = *reinterpret_cast<SmallSmem<STAGES> *>(small_smem_raw);
    const int64_t m0 = int64_t(blockIdx.x) * kSmBM, n0 = int64_t(blockIdx.y) * kSmBN;
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int64_t chunks = (K + kSmKC - 1) / kSmKC;

    // copy plan
    int64_t aoff[kRA], boff[kRB];
    uint32_t adst[kRA], bdst[kRB];
    int alim[kRA], blim[kRB];   // the element's k in the chunk, or kSmKC past M / N
#pragma unroll
    for (int r = 0; r < kRA; ++r) {
        const int e = tid + r * kSmThreads;
        const int i = transA ? e % kSmBM : e / kSmKC;
        const int k = transA ? e / kSmBM : e % kSmKC;
        const int64_t gi = m0 + i;
        alim[r] = gi < M ? k : kSmKC;
        aoff[r] = transA ? int64_t(k) * lda + gi : gi * lda + k;
        adst[r] = smem_addr(&sm.a[0][k][i]);
    }
#pragma unroll
    for (int r = 0; r < kRB; ++r) {
        const int e = tid + r * kSmThreads;
        const int j = transB ? e / kSmKC : e % kSmBN;
        const int k = transB ? e % kSmKC : e / kSmBN;
        const int64_t gj = n0 + j;
        blim[r] = gj < N ? k : kSmKC;
        boff[r] = transB ? gj * ldb + k : int64_t(k) * ldb + gj;
        bdst[r] = smem_addr(&sm.b[0][k][j]);
    }
    const int64_t ainc = transA ? int64_t(kSmKC) * lda : kSmKC;
    const int64_t binc = transB ? int64_t(kSmKC) : int64_t(kSmKC) * ldb;
    constexpr uint32_t kStageA = sizeof(sm.a[0]), kStageB = sizeof(sm.b[0]);

    auto stage = [&](int s, int64_t c) {
        const int64_t left = K - c * kSmKC;
        const int kr = left < kSmKC ? int(left) : kSmKC;   // k's of this chunk inside K
        const float *Ac = A + c * ainc, *Bc = B + c * binc;
#pragma unroll
        for (int r = 0; r < kRA; ++r) {
            const bool ok = alim[r] < kr && REPOPS_DBG_OK(dbg.a, Ac + aoff[r], 4, dbg.status);
            cp_async_4_to(adst[r] + s * kStageA, ok ? Ac + aoff[r] : A, ok ? 4u : 0u);
        }
#pragma unroll
        for (int r = 0; r < kRB; ++r) {
            const bool ok = blim[r] < kr && REPOPS_DBG_OK(dbg.b, Bc + boff[r], 4, dbg.status);
            cp_async_4_to(bdst[r] + s * kStageB, ok ? Bc + boff[r] : B, ok ? 4u : 0u);
        }
    };

    // ring: chunk c lives in stage c % STAGES; one commit group per chunk
    // (possibly empty past the last chunk, so the wait count stays fixed)
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < chunks) stage(s, s);
        cp_async_commit();
    }
    u64 acc0 = pack2(0.0f, 0.0f);   // row 2ty,     columns 2tx, 2tx + 1
    u64 acc1 = pack2(0.0f, 0.0f);   // row 2ty + 1, columns 2tx, 2tx + 1
    int s = 0;                      // stage of chunk c
    for (int64_t c = 0; c < chunks; ++c) {
        cp_async_wait<STAGES - 2>();   // chunk c has landed (this thread's copies)
        __syncthreads();               // ... and every thread's; stage (c - 1) % STAGES is free
        const int64_t next = c + STAGES - 1;
        if (next < chunks) stage(s == 0 ? STAGES - 1 : s - 1, next);
        cp_async_commit();
#pragma unroll
        for (int k = 0; k < kSmKC; ++k) {
            const float2 a = *reinterpret_cast<const float2 *>(&sm.a[s][k][2 * ty]);
            const float2 b = *reinterpret_cast<const float2 *>(&sm.b[s][k][2 * tx]);
            acc0 = fold2(acc0, a.x, b.x, a.x, b.y);
            acc1 = fold2(acc1, a.y, b.x, a.y, b.y);
        }
        s = s == STAGES - 1 ? 0 : s + 1;
    }
    cp_async_wait<0>();

    float c00, c01, c10, c11;
    unpack2(acc0, c00, c01);
    unpack2(acc1, c10, c11);
    const int64_t i0 = m0 + 2 * ty, j0 = n0 + 2 * tx;
    auto put = [&](int64_t i, int64_t j, float v) {
        if (i < M && j < N && REPOPS_DBG_OK(dbg.c, C + i * ldc + j, 4, dbg.status)) C[i * ldc + j] = v;
    };
    put(i0, j0, c00);
    put(i0, j0 + 1, c01);
    put(i0 + 1, j0, c10);
    put(i0 + 1, j0 + 1, c11);
}

constexpr int kSmStages = 3;

}  // namespace

int gemm_small_launch(const GemmProblem &p) {
    const int64_t gm = (p.M + kSmBM - 1) / kSmBM, gn = (p.N + kSmBN - 1) / kSmBN;
    if (gm > 0x7fffffffLL || gn > 65535) return REPOPS_ERR_UNSUPPORTED;
    constexpr int smem = int(sizeof(SmallSmem<kSmStages>));
    static_assert(smem <= 48 * 1024, "the ring fits the default dynamic shared memory limit");
    auto kern = gemm_small_kernel<kSmStages>;
    SmallDbg dbg;
    dbg.a.lo = p.span_a[0]; dbg.a.hi = p.span_a[1];
    dbg.b.lo = p.span_b[0]; dbg.b.hi = p.span_b[1];
    dbg.c.lo = p.span_c[0]; dbg.c.hi = p.span_c[1];
    dbg.status = p.status;
    kern<<<dim3(unsigned(gm), unsigned(gn)), kSmThreads, smem, p.stream>>>(
        p.transA, p.transB, p.M, p.N, p.K, p.A, p.lda, p.B, p.ldb, p.C, p.ldc, dbg);
    return check_launch();
}

}  // namespace repops
