// GEMM tile configuration 3: CTA tile 64x64, 128 threads, 8x4 per thread, 3 stages.
// One configuration per translation unit so the library compiles in parallel.
#include "gemm_kernels.cuh"

namespace {
using Cfg3 = repops::gemm::Tile<8,4,2,2,3>;
}
REPOPS_DEFINE_GEMM_CONFIG(3, Cfg3)
