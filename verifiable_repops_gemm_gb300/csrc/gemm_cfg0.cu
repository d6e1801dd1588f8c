// GEMM tile configuration 0: CTA tile 128x128, 256 threads, 8x8 per thread, 4 stages.
// One configuration per translation unit so the library compiles in parallel.
#include "gemm_kernels.cuh"

namespace {
using Cfg0 = repops::gemm::Tile<8,8,4,2,4>;
}
REPOPS_DEFINE_GEMM_CONFIG(0, Cfg0)
