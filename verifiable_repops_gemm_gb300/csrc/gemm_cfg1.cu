// GEMM tile configuration 1: CTA tile 64x128, 128 threads, 8x8 per thread, 4 stages.
// One configuration per translation unit so the library compiles in parallel.
#include "gemm_kernels.cuh"

namespace {
using Cfg1 = repops::gemm::Tile<8,8,2,2,4>;
}
REPOPS_DEFINE_GEMM_CONFIG(1, Cfg1)
