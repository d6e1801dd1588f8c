// GEMM tile configuration 4: CTA tile 32x64, 128 threads, 4x4 per thread, 3 stages.
// One configuration per translation unit so the library compiles in parallel.
#include "gemm_kernels.cuh"

namespace {
using Cfg4 = repops::gemm::Tile<4,4,2,2,3>;
}
REPOPS_DEFINE_GEMM_CONFIG(4, Cfg4)
