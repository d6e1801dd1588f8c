// GEMM tile configuration 2: CTA tile 128x64, 128 threads, 8x8 per thread, 4 stages.
// One configuration per translation unit so the library compiles in parallel.
#include "gemm_kernels.cuh"

namespace {
using Cfg2 = repops::gemm::Tile<8,8,4,1,4>;
}
REPOPS_DEFINE_GEMM_CONFIG(2, Cfg2)
