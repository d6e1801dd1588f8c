// gemm_common.h -- host-side description of one GEMM call and of the tile
// configurations compiled into the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace repops {

struct GemmProblem {
    int transA = 0, transB = 0;
    int64_t M = 0, N = 0, K = 0;
    const float *A = nullptr;
    int64_t lda = 0;
    const float *B = nullptr;
    int64_t ldb = 0;
    float *C = nullptr;
    int64_t ldc = 0;
    cudaStream_t stream = nullptr;
    unsigned *status = nullptr;   // device address of the sticky status word
    // Batched / fused-epilogue form (repops_gemm_f32_batched).  ex == false is
    // the plain GEMM and ignores the fields below.
    bool ex = false;
    int64_t batch = 1;
    int64_t strideA = 0, strideB = 0, strideC = 0;   // elements; 0 = shared by every batch
    float alpha = 1.0f;
    const float *bias = nullptr;                      // N values, or null
    int act = 0;                                      // 0 none, 1 GeLU
    const float *R = nullptr;                         // residual, or null
    int64_t ldr = 0, strideR = 0;
    int64_t causal = -1;   // >= 0: tiles wholly above j = causal + i are skipped
    int64_t k_lo = -1;     // >= 0: row i's k-chain starts at max(0, i - k_lo)
    int64_t k_hi = -1;     // >= 0: row i's k-chain ends at min(K - 1, i + k_hi)
    int64_t b_group = 1;   // batch b reads B_(b / b_group)
    // Chained k-split (TMA loader, batch 1, no causal skip or band): a
    // persistent grid of sk_workers CTAs; sk_scratch holds their heads'
    // accumulators and flags (gemm_sk_scratch_cfg<N>, flags zeroed).  0 = one
    // CTA per tile.
    int sk_workers = 0;
    void *sk_scratch = nullptr;
    // Spans of A, B and C the checked build tests every access against
    // (filled by the dispatchers; unused in the release build).
    uintptr_t span_a[2] = {0, 0}, span_b[2] = {0, 0}, span_c[2] = {0, 0};
};

struct GemmConfigInfo {
    int bm, bn, threads, tm, tn, stages;
};

// One entry per compiled configuration; defined in gemm_cfg<N>.cu.
using GemmLauncher = int (*)(const GemmProblem &, int loader);
using GemmOccupancy = int (*)();   // resident CTAs per SM (TMA kernel), current device

#define REPOPS_DECLARE_GEMM_CONFIG(N)          \
    int gemm_launch_cfg##N(const GemmProblem &, int); \
    int gemm_occupancy_cfg##N();               \
    GemmConfigInfo gemm_info_cfg##N();         \
    size_t gemm_sk_scratch_cfg##N(int workers);

REPOPS_DECLARE_GEMM_CONFIG(0)
REPOPS_DECLARE_GEMM_CONFIG(1)
REPOPS_DECLARE_GEMM_CONFIG(2)
REPOPS_DECLARE_GEMM_CONFIG(3)
REPOPS_DECLARE_GEMM_CONFIG(4)

constexpr int kGemmConfigCount = 5;

// True when the TMA loader can serve this problem (alignment, extents).
bool gemm_tma_eligible(const GemmProblem &p);

// The small-output kernel (gemm_small.cu): plain GEMM only (p.ex false).
int gemm_small_launch(const GemmProblem &p);

}  // namespace repops
