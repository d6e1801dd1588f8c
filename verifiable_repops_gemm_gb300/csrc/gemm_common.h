// gemm_common.h -- host-side description of one GEMM call and of the tile
// configurations compiled into the library.
#pragma once

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
    GemmConfigInfo gemm_info_cfg##N();

REPOPS_DECLARE_GEMM_CONFIG(0)
REPOPS_DECLARE_GEMM_CONFIG(1)
REPOPS_DECLARE_GEMM_CONFIG(2)
REPOPS_DECLARE_GEMM_CONFIG(3)
REPOPS_DECLARE_GEMM_CONFIG(4)

constexpr int kGemmConfigCount = 5;

// True when the TMA loader can serve this problem (alignment, extents).
bool gemm_tma_eligible(const GemmProblem &p);

}  // namespace repops
