// gemm.cu -- C-ABI entry points of the order-fixed FP32 GEMM: argument checks,
// choice of tile configuration and loader, the sticky device status word.
//
// The arithmetic itself is in gemm_kernels.cuh ("Verde与RepOps" §3.2 matmul
// example; §3.1: the bits must not depend on core count, tiling or strides).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "gemm_common.h"
#include "gemm_kernels.cuh"
#include "internal.cuh"

namespace repops {

namespace {

// Sticky status word: bit 0 = a TMA wait gave up.  One per device (a
// __device__ variable exists once per device that loads the library), shared
// by every caller that has not bound a word of its own.
__device__ unsigned g_gemm_status;

// The caller's own status word for this host thread's launches
// (repops_set_thread_status_word), or null for the shared one.
thread_local unsigned *t_status_word = nullptr;

constexpr int kMaxDevices = 64;

// The shared word's device address, looked up once per device and context: a
// symbol's address is only valid in the context it was looked up in, so a new
// context (after cudaDeviceReset, say) looks it up again.
struct StatusAddr {
    std::mutex mu;
    uint64_t ctx_key = 0;
    unsigned *addr = nullptr;
};
StatusAddr g_status_addr[kMaxDevices];

int shared_status_address(unsigned **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return REPOPS_ERR_UNSUPPORTED;
    uint64_t key = 0;
    int rc = current_context_key(&key);
    if (rc != REPOPS_OK) return rc;
    StatusAddr &s = g_status_addr[dev];
    std::lock_guard<std::mutex> lock(s.mu);
    if (s.ctx_key != key || !s.addr) {
        unsigned *p = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_gemm_status);
        if (e != cudaSuccess) return set_cuda_error(e);
        s.addr = p;
        s.ctx_key = key;
    }
    *out = s.addr;
    return REPOPS_OK;
}

// The word the kernels this thread launches report into.
int status_address(unsigned **out) {
    if (t_status_word) {
        *out = t_status_word;
        return REPOPS_OK;
    }
    return shared_status_address(out);
}

}  // namespace

int status_word_address(unsigned **out) { return status_address(out); }

namespace {

// Failure-detection self-test: thread 0 waits on a phase of an mbarrier that
// nothing will complete, gives up after limit_ns and sets the sticky status
// word, exactly as a GEMM wait that timed out would.  Nothing else is touched.
__global__ void bounded_wait_selftest_kernel(unsigned *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait_bounded_ns(&bar, 0u, limit_ns)) atomicOr(status, 1u);
}

// The flag of the second self-test: zero, and nothing ever sets it.
__device__ unsigned g_selftest_flag;

// Failure-detection self-test of the chained split's wait: thread 0 waits for
// a flag that nothing sets (the wait a tail makes for its head's partial
// sums), gives up after limit_ns and sets the sticky status word.
__global__ void flag_wait_selftest_kernel(unsigned *status, uint64_t limit_ns) {
    if (threadIdx.x != 0) return;
    if (!gemm::flag_wait_bounded_ns(&g_selftest_flag, limit_ns)) atomicOr(status, 1u);
}

const GemmLauncher kLaunch[kGemmConfigCount] = {gemm_launch_cfg0, gemm_launch_cfg1, gemm_launch_cfg2,
                                                gemm_launch_cfg3, gemm_launch_cfg4};
const GemmOccupancy kOccupancy[kGemmConfigCount] = {gemm_occupancy_cfg0, gemm_occupancy_cfg1,
                                                    gemm_occupancy_cfg2, gemm_occupancy_cfg3,
                                                    gemm_occupancy_cfg4};
using GemmSkScratch = size_t (*)(int);
const GemmSkScratch kSkScratch[kGemmConfigCount] = {gemm_sk_scratch_cfg0, gemm_sk_scratch_cfg1,
                                                    gemm_sk_scratch_cfg2, gemm_sk_scratch_cfg3,
                                                    gemm_sk_scratch_cfg4};
GemmConfigInfo config_info(int c) {
    switch (c) {
        case 0: return gemm_info_cfg0();
        case 1: return gemm_info_cfg1();
        case 2: return gemm_info_cfg2();
        case 3: return gemm_info_cfg3();
        default: return gemm_info_cfg4();
    }
}

// Resident CTAs per SM for each configuration, cached per device.
std::atomic<int> g_occ[kMaxDevices][kGemmConfigCount];

int occupancy_of(int dev, int c) {
    int v = g_occ[dev][c].load(std::memory_order_relaxed);
    if (v == 0) {
        v = std::max(1, kOccupancy[c]());
        g_occ[dev][c].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Per-tile throughput of a configuration relative to the 64x128 / 128x64
// tiles (8x8 accumulators, 128 consumer threads), fitted to measurements of
// all five configurations on 20 shapes from 256^3 to 8192^3 on a GB300.  The
// 128x128 tile's figure sits just under 1: where the two tiles' waves line up
// they are within 1% either way, and 64x128 is the faster at 8192^3.
double relative_efficiency(const GemmConfigInfo &ci) {
    const int acc = ci.tm * ci.tn;
    if (acc >= 64) return ci.threads > 128 ? 0.995 : 1.0;
    if (acc >= 32) return 0.94;
    return 0.76;
}

// Picks the configuration with the smallest modelled time.  The busiest SM
// runs n = ceil(tiles / SMs) tiles, `conc` at a time; a tile takes
// BM * BN / eff when `conc` share the SM, and a last round with fewer tiles
// than `conc` is charged 0.7 of a shared round (a lone CTA runs faster than
// half speed).  An SM with fewer resident consumer warps than it needs to hide
// the ring's fill and the epilogue is modelled as proportionally slower -- 8
// warps for long k-chains, more as K shrinks below 256.  Fitted to the same
// measurements: its choice is within 2% of the fastest configuration on all
// 20 shapes and within 1% on 19 (the previous round-based model lost up to 9%).
//
// With `allow_sk`, each configuration whose tiles outnumber its resident CTAs
// is also costed with the chained k-split (every SM gets tiles / SMs tiles'
// worth of k-slices, plus 2% for the heads' stores and loads), and *sk tells
// whether that schedule won.  Persistent CTAs run as fast as one-tile CTAs
// when one fills an SM (128 x 128, 8 consumer warps: 34.9 against 35.1
// TFLOP/s at 8192^3, where nothing is left to balance), but two persistent
// CTAs sharing an SM measured 7% slower than two one-tile CTAs (32.8 against
// 35.2 for 64 x 128), so those are charged 1/0.93.
int choose_plan(int64_t M, int64_t N, int64_t K, int64_t batch, bool allow_sk, bool *sk) {
    if (sk) *sk = false;
    DeviceInfo di;
    if (current_device_info(&di) != REPOPS_OK || di.device < 0 || di.device >= kMaxDevices) return 0;
    double best_t = 0;
    int best = 0;
    bool best_sk = false;
    for (int c = 0; c < kGemmConfigCount; ++c) {
        const GemmConfigInfo ci = config_info(c);
        const double tiles =
            double((M + ci.bm - 1) / ci.bm) * double((N + ci.bn - 1) / ci.bn) * double(std::max<int64_t>(batch, 1));
        const double n = std::ceil(tiles / di.sms);
        const double conc = std::max(1, occupancy_of(di.device, c));
        const double full = std::floor(n / conc), rem = n - full * conc;
        const double warps = std::min(conc, n) * ci.threads / 32.0;
        const double need = std::min(32.0, 8.0 * std::max(1.0, 256.0 / double(std::max<int64_t>(K, 1))));
        const double eff = relative_efficiency(ci) * std::min(1.0, warps / need);
        const double t = (full * conc + (rem > 0 ? 0.7 * conc : 0.0)) * double(ci.bm) * double(ci.bn) / eff;
        if (c == 0 || t < best_t * 0.999) { best_t = t; best = c; best_sk = false; }
        if (allow_sk && tiles >= conc * di.sms) {
            const double eff_sk = relative_efficiency(ci) * std::min(1.0, conc * ci.threads / 32.0 / need);
            const double shared_sm = conc > 1 ? 1.0 / 0.93 : 1.0;
            const double t_sk = 1.02 * shared_sm * tiles / di.sms * double(ci.bm) * double(ci.bn) / eff_sk;
            if (t_sk < best_t * 0.999) { best_t = t_sk; best = c; best_sk = true; }
        }
    }
    if (sk) *sk = best_sk;
    return best;
}

// Tile choice for a banded product (k_lo / k_hi set): the tiles' k-ranges
// differ -- a tile runs the whole 32-k slices covering its rows' bands -- so
// the time is modelled as the longer of the longest tile (sharing its SM with
// the other resident CTAs) and the total work spread over the SMs.  For the
// per-head attention gradients (2048 x 64 outputs, 8 batches, band k >= i)
// it picks the 32 x 64 tile, measured 18% faster than the 64 x 64 one the
// unbanded model takes.
int choose_config_banded(int64_t M, int64_t N, int64_t K, int64_t batch, int64_t k_lo, int64_t k_hi) {
    DeviceInfo di;
    if (current_device_info(&di) != REPOPS_OK || di.device < 0 || di.device >= kMaxDevices) return 0;
    double best_t = 0;
    int best = 0;
    for (int c = 0; c < kGemmConfigCount; ++c) {
        const GemmConfigInfo ci = config_info(c);
        const double eff = relative_efficiency(ci), conc = std::max(1, occupancy_of(di.device, c));
        double longest = 0, total = 0;
        for (int64_t m0 = 0; m0 < M; m0 += ci.bm) {
            const int64_t lo = k_lo >= 0 ? std::max<int64_t>(0, m0 - k_lo) : 0;
            const int64_t hi = k_hi >= 0 ? std::min<int64_t>(K, m0 + ci.bm + k_hi) : K;
            const double slices = lo < hi ? double((hi + 31) / 32 - lo / 32) : 0.0;
            const double w = double(ci.bm) * double(ci.bn) * slices / eff;
            longest = std::max(longest, w);
            total += w;
        }
        total *= double((N + ci.bn - 1) / ci.bn) * double(std::max<int64_t>(batch, 1));
        const double t = std::max(longest * conc, total / di.sms);
        if (c == 0 || t < best_t * 0.999) { best_t = t; best = c; }
    }
    return best;
}

// Span in elements of a rows x cols operand with leading dimension ld.
bool operand_span(int64_t rows, int64_t cols, int64_t ld, uint64_t *bytes) {
    if (rows == 0 || cols == 0) { *bytes = 0; return true; }
    // (rows - 1) * ld + cols must fit in int64 (element index)
    if (rows - 1 > (INT64_MAX - cols) / std::max<int64_t>(ld, 1)) return false;
    const int64_t elems = (rows - 1) * ld + cols;
    if (elems > INT64_MAX / 4) return false;
    *bytes = uint64_t(elems) * 4u;
    return true;
}

// The spans of the caller's operands, for the checked build's access tests.
void set_spans(GemmProblem &p, uint64_t a_bytes, uint64_t b_bytes, uint64_t c_bytes) {
    p.span_a[0] = reinterpret_cast<uintptr_t>(p.A);
    p.span_a[1] = p.span_a[0] + a_bytes;
    p.span_b[0] = reinterpret_cast<uintptr_t>(p.B);
    p.span_b[1] = p.span_b[0] + b_bytes;
    p.span_c[0] = reinterpret_cast<uintptr_t>(p.C);
    p.span_c[1] = p.span_c[0] + c_bytes;
}

__global__ void fill_positive_zero(float *C, int64_t M, int64_t N, int64_t ldc) {
    const int64_t total = M * N;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e - i * N;
        C[i * ldc + j] = 0.0f;
    }
}

// Copies a rows x cols row-major block from pitch ld_src to pitch ld_dst
// (elements).  A pure copy: the GEMM reads the same values in the same order.
__global__ void repack_rows(const float *__restrict__ src, int64_t ld_src, float *__restrict__ dst,
                            int64_t ld_dst, int64_t rows, int64_t cols) {
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const float *s = src + r * ld_src;
        float *d = dst + r * ld_dst;
        for (int64_t c = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; c < cols;
             c += int64_t(gridDim.x) * blockDim.x)
            d[c] = s[c];
    }
}

// dst = src^T: src is rows x cols at pitch lds, dst cols x rows at pitch ldd.
// 32 x 32 tiles through shared memory (one pad column: conflict-free), so
// both the reads and the writes are coalesced.  A pure copy.
__global__ void __launch_bounds__(256)
transpose_kernel(const float *__restrict__ src, int64_t lds, float *__restrict__ dst, int64_t ldd, int64_t rows,
                 int64_t cols) {
    __shared__ float tile[32][33];
    for (int64_t by = blockIdx.y; by * 32 < rows; by += gridDim.y) {
        for (int64_t bx = blockIdx.x; bx * 32 < cols; bx += gridDim.x) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t r = by * 32 + threadIdx.y + 8 * i, c = bx * 32 + threadIdx.x;
                if (r < rows && c < cols) tile[threadIdx.y + 8 * i][threadIdx.x] = src[r * lds + c];
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t r = bx * 32 + threadIdx.y + 8 * i, c = by * 32 + threadIdx.x;
                if (r < cols && c < rows) dst[r * ldd + c] = tile[threadIdx.x][threadIdx.y + 8 * i];
            }
            __syncthreads();
        }
    }
}

int launch_transpose(const float *src, int64_t lds, int64_t rows, int64_t cols, float *dst, int64_t ldd,
                     cudaStream_t stream) {
    const dim3 grid(unsigned(std::min<int64_t>((cols + 31) / 32, 65535)),
                    unsigned(std::min<int64_t>((rows + 31) / 32, 65535)));
    transpose_kernel<<<grid, dim3(32, 8), 0, stream>>>(src, lds, dst, ldd, rows, cols);
    return check_launch();
}

// Work (2*M*N*K) from which repacking TMA-incompatible operands pays off: the
// copy streams each operand once (~10-20 us for the ragged 4097x1023x3001
// workload) and lets the TMA kernels run instead of the 4-byte loader.  The
// same bound holds for transposing a row-major A into the M-inner layout.
constexpr double kRepackMinFlops = 4.0e9;
// A B stored transposed (K-inner) is transposed from 1 GFLOP on: measured on
// a GB300 (L2 flushed, synchronised after each call), 1024^3 20.4 -> 21.7,
// 1024 x 1024 x 1536 21.2 -> 23.3 and 2048 x 1024 x 512 21.2 -> 22.9 TFLOP/s;
// 768^3 (0.9 GFLOP) 18.2 -> 17.5, slower.  Transposing A pays only from
// kRepackMinFlops: at 1024^3 it measured 23.1 -> 22.9.
constexpr double kTransposeBMinFlops = 1.0e9;

bool operand_tma_ready(const float *ptr, int64_t ld) {
    return reinterpret_cast<uintptr_t>(ptr) % 16 == 0 && ld % 4 == 0;
}

int launch_repack(const float *src, int64_t ld_src, float *dst, int64_t ld_dst, int64_t rows, int64_t cols,
                  cudaStream_t stream) {
    const int threads = 256;
    const int64_t gx = std::min<int64_t>((cols + threads - 1) / threads, 64);
    const int64_t gy = std::min<int64_t>(rows, 65535);
    repack_rows<<<dim3(unsigned(gx), unsigned(gy)), threads, 0, stream>>>(src, ld_src, dst, ld_dst, rows, cols);
    return check_launch();
}

// Bytes of the copy copy_operand makes of a rows x cols operand.
uint64_t copy_operand_bytes(int64_t rows, int64_t cols, bool transpose) {
    const int64_t outer = transpose ? cols : rows, inner = transpose ? rows : cols;
    return uint64_t(outer) * uint64_t((inner + 3) / 4 * 4) * 4u;
}

// Copies a rows x cols operand (pitch ld) into scratch with a 16-byte pitch:
// transposed (cols x rows) when `transpose`, else as it is.  The scratch is
// `pre` (the caller's workspace, copy_operand_bytes bytes) or, when that is
// null, stream-ordered memory from the pool that the caller releases.  *out
// is the scratch (null, and REPOPS_OK, when the allocation is refused: the
// caller then keeps its operand) and *pitch its row pitch in elements.
int copy_operand(const float *src, int64_t ld, int64_t rows, int64_t cols, bool transpose, cudaStream_t stream,
                 void **out, int64_t *pitch, void *pre = nullptr) {
    const int64_t inner = transpose ? rows : cols;
    const int64_t pm = (inner + 3) / 4 * 4;
    *out = pre;
    if (!pre && scratch_malloc(out, size_t(copy_operand_bytes(rows, cols, transpose)), stream) != cudaSuccess) {
        cudaGetLastError();   // a refused allocation is not an error here
        *out = nullptr;
        return REPOPS_OK;
    }
    float *dst = static_cast<float *>(*out);
    const int rc = transpose ? launch_transpose(src, ld, rows, cols, dst, pm, stream)
                             : launch_repack(src, ld, dst, pm, rows, cols, stream);
    if (rc != REPOPS_OK) {
        if (!pre) cudaFreeAsync(*out, stream);
        *out = nullptr;
        return rc;
    }
    *pitch = pm;
    return REPOPS_OK;
}

// The small-output kernel (16 x 32 CTA tiles) runs outputs of at most
// 196,608 elements, where the tiled kernels leave most SMs idle; measured
// crossover on GB300 between 384^2 (small kernel 8.4 us, tiled 13.1 us) and
// 512^2 (18.8 against 16.9 us).
constexpr int64_t kSmallMaxOutputs = 3 << 16;

bool small_output(int64_t M, int64_t N, int64_t K) {
    return M > 0 && N > 0 && K > 0 && M * N <= kSmallMaxOutputs && N <= 65535LL * 32;
}

// Chained k-split request of a call: kSkAuto lets the automatic choice decide
// (config -1 and the automatic loader only), a value >= 0 asks for it with
// that many workers (0 = every resident CTA slot), and any other negative
// value never splits.
constexpr int kSkAuto = -1;

// Workers and scratch bytes (the heads' accumulators, then the flags) of a
// chained k-split of an M x N output on configuration cfg with `req` workers
// (0 = every resident slot, at most one per tile).  REPOPS_ERR_UNSUPPORTED
// when it cannot run with that many.
int chained_split_shape(int64_t M, int64_t N, int cfg, int req, int *workers, uint64_t *bytes) {
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != REPOPS_OK) return rc;
    const GemmConfigInfo ci = config_info(cfg);
    const int64_t tiles = ((M + ci.bm - 1) / ci.bm) * ((N + ci.bn - 1) / ci.bn);
    const int64_t slots = int64_t(occupancy_of(di.device, cfg)) * di.sms;
    const int64_t w = req == 0 ? std::min<int64_t>(slots, tiles) : req;
    if (w < 1 || w > slots || w > tiles) return REPOPS_ERR_UNSUPPORTED;
    *workers = int(w);
    *bytes = kSkScratch[cfg](int(w));
    return REPOPS_OK;
}

// Runs p with the chained k-split on `workers` persistent CTAs of configuration
// cfg (0 = every resident slot, at most one per tile): scratch for the heads'
// accumulators and flags (`pre`, the caller's workspace, or stream-ordered
// memory from the pool), the flags zeroed, the launch, pool scratch released.
// REPOPS_ERR_UNSUPPORTED when the split cannot run (the caller then runs the
// one-tile-per-CTA kernel): no TMA, too many workers, or a refused allocation.
int launch_chained_split(GemmProblem p, int cfg, int workers, void *pre = nullptr) {
    uint64_t bytes = 0;
    int rc = chained_split_shape(p.M, p.N, cfg, workers, &workers, &bytes);
    if (rc != REPOPS_OK) return rc;
    const size_t flag_bytes = size_t(workers) * size_t(config_info(cfg).threads) * 4u;
    void *scratch = pre;
    if (!pre && scratch_malloc(&scratch, size_t(bytes), p.stream) != cudaSuccess) {
        cudaGetLastError();
        return REPOPS_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaMemsetAsync(static_cast<unsigned char *>(scratch) + (bytes - flag_bytes), 0, flag_bytes,
                                    p.stream);
    if (e != cudaSuccess) {
        if (!pre) cudaFreeAsync(scratch, p.stream);
        return set_cuda_error(e);
    }
    p.sk_workers = workers;
    p.sk_scratch = scratch;
    rc = kLaunch[cfg](p, REPOPS_LOADER_TMA);
    if (!pre) {
        e = cudaFreeAsync(scratch, p.stream);
        if (rc == REPOPS_OK && e != cudaSuccess) rc = set_cuda_error(e);
    }
    return rc;
}

inline uint64_t round_up_256(uint64_t x) { return (x + 255) / 256 * 256; }

// The GEMM's dispatch.  Scratch (operand copies, chained-split accumulators)
// comes from `ws` (ws_bytes bytes, 256-byte aligned) when it is large enough
// for the whole plan, else from the pool.  With need_out set nothing is
// launched: *need_out receives the bytes of scratch the plan takes (0 when it
// runs on the caller's operands alone), and C is not looked at.
int gemm_dispatch(int config, int loader, int transA, int transB, int64_t M, int64_t N, int64_t K,
                  const float *A, int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc,
                  cudaStream_t stream, int sk_req = kSkAuto, void *ws = nullptr, uint64_t ws_bytes = 0,
                  uint64_t *need_out = nullptr) {
    if (need_out) *need_out = 0;
    if (M < 0 || N < 0 || K < 0) return REPOPS_ERR_INVALID_ARG;
    if (config < -1 || config >= kGemmConfigCount) return REPOPS_ERR_INVALID_ARG;
    if (loader != REPOPS_LOADER_AUTO && loader != REPOPS_LOADER_TMA && loader != REPOPS_LOADER_CPASYNC &&
        loader != REPOPS_LOADER_DIRECT)
        return REPOPS_ERR_INVALID_ARG;
    const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;
    if (lda < std::max<int64_t>(1, a_cols) || ldb < std::max<int64_t>(1, b_cols) ||
        ldc < std::max<int64_t>(1, N))
        return REPOPS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return REPOPS_OK;
    if (!C && !need_out) return REPOPS_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B)) return REPOPS_ERR_INVALID_ARG;
    uint64_t a_bytes = 0, b_bytes = 0, c_bytes = 0;
    if (!operand_span(a_rows, a_cols, lda, &a_bytes) || !operand_span(b_rows, b_cols, ldb, &b_bytes) ||
        !operand_span(M, N, ldc, &c_bytes))
        return REPOPS_ERR_INVALID_ARG;
    if (!need_out && (ranges_overlap(C, c_bytes, A, a_bytes) || ranges_overlap(C, c_bytes, B, b_bytes)))
        return REPOPS_ERR_ALIAS;
    if (ws && !need_out) {
        if (reinterpret_cast<uintptr_t>(ws) % 256) return REPOPS_ERR_INVALID_ARG;
        if (ranges_overlap(ws, ws_bytes, A, a_bytes) || ranges_overlap(ws, ws_bytes, B, b_bytes) ||
            ranges_overlap(ws, ws_bytes, C, c_bytes))
            return REPOPS_ERR_ALIAS;
    }

    if (K == 0) {
        if (need_out) return REPOPS_OK;
        const int64_t total = M * N;
        const int threads = 256;
        const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, 65536);
        fill_positive_zero<<<int(blocks), threads, 0, stream>>>(C, M, N, ldc);
        return check_launch();
    }

    GemmProblem p;
    p.transA = transA ? 1 : 0;
    p.transB = transB ? 1 : 0;
    p.M = M; p.N = N; p.K = K;
    p.A = A; p.lda = lda; p.B = B; p.ldb = ldb; p.C = C; p.ldc = ldc;
    p.stream = stream;
    set_spans(p, a_bytes, b_bytes, c_bytes);
    int rc = status_address(&p.status);
    if (rc != REPOPS_OK) return rc;
    const bool sk_explicit = sk_req >= 0;
    if (!sk_explicit &&
        (loader == REPOPS_LOADER_DIRECT || (loader == REPOPS_LOADER_AUTO && config < 0 && small_output(M, N, K))))
        return need_out ? REPOPS_OK : gemm_small_launch(p);

    bool sk_auto = false;
    const int cfg = config >= 0 ? config
                                : choose_plan(M, N, K, 1, sk_req == kSkAuto && loader == REPOPS_LOADER_AUTO,
                                              &sk_auto);
    const bool want_sk = sk_explicit || sk_auto;
    bool tma_ok = gemm_tma_eligible(p);
    if ((loader == REPOPS_LOADER_TMA || sk_explicit) && !tma_ok) return REPOPS_ERR_UNSUPPORTED;

    // Large problems (automatic loader) run on stream-ordered scratch copies
    // where that is faster; the kernels then compute the same products and
    // sums in the same order, so the bits do not change:
    //  - B stored transposed (K-inner, the slowest layout: 0.78 of the FP32
    //    pipe at 8192^3) is transposed into a row-major B with a 16-byte pitch
    //    (from 1 GFLOP; the other copies from 4 GFLOP);
    //  - A stored row-major (K-inner) is transposed into an M-inner A: those
    //    kernels (products paired along m) run 3% faster at 8192^3 (35.1
    //    against 34.0 TFLOP/s);
    //  - an operand TMA cannot describe otherwise (a base not 16-byte aligned,
    //    a leading dimension not a multiple of 4) is repacked with a 16-byte
    //    pitch, so that the TMA kernels run instead of the 4-byte loader.
    // Each copy streams its operand once (~0.1 ms for 8192^2).  Without the
    // scratch (a refused allocation) the caller's operands are used as they are.
    const double flops = 2.0 * double(M) * double(N) * double(K);
    const bool large = loader == REPOPS_LOADER_AUTO && flops >= kRepackMinFlops;
    const bool transpose_b = loader == REPOPS_LOADER_AUTO && p.transB && flops >= kTransposeBMinFlops;
    const bool copy_b = transpose_b || (large && !operand_tma_ready(p.B, p.ldb));
    const bool copy_a = large && (!p.transA || !operand_tma_ready(p.A, p.lda));
    // The plan's scratch: the copies (A M-inner, B N-inner, 16-byte pitches),
    // then the chained split's accumulators when it runs on those operands.
    const uint64_t need_a = copy_a ? copy_operand_bytes(K, M, false) : 0;
    const uint64_t need_b = copy_b ? copy_operand_bytes(K, N, false) : 0;
    uint64_t need_sk = 0;
    if (want_sk && loader != REPOPS_LOADER_CPASYNC) {
        GemmProblem q = p;   // the operands as the kernels will see them (any 16-byte aligned base)
        const float *aligned = reinterpret_cast<const float *>(uintptr_t(256));
        if (copy_a) { q.A = aligned; q.lda = (M + 3) / 4 * 4; q.transA = 1; }
        if (copy_b) { q.B = aligned; q.ldb = (N + 3) / 4 * 4; q.transB = 0; }
        int workers = 0;
        if (!gemm_tma_eligible(q) ||
            chained_split_shape(M, N, cfg, sk_explicit ? sk_req : 0, &workers, &need_sk) != REPOPS_OK)
            need_sk = 0;
    }
    const uint64_t need = round_up_256(need_a) + round_up_256(need_b) + round_up_256(need_sk);
    if (need_out) {
        *need_out = need;
        return REPOPS_OK;
    }
    // carved from the caller's workspace when it holds the whole plan
    unsigned char *wsp = (ws && need > 0 && ws_bytes >= need) ? static_cast<unsigned char *>(ws) : nullptr;
    void *pre_a = wsp, *pre_b = wsp ? wsp + round_up_256(need_a) : nullptr;
    void *pre_sk = wsp ? wsp + round_up_256(need_a) + round_up_256(need_b) : nullptr;
    void *bscratch = nullptr, *ascratch = nullptr;
    auto fail = [&](int code) {
        if (bscratch && !pre_b) cudaFreeAsync(bscratch, stream);
        if (ascratch && !pre_a) cudaFreeAsync(ascratch, stream);
        return code;
    };
    if (copy_b) {
        // B stored transposed (N x K) is transposed, an unaligned row-major B repacked
        int64_t pitch = 0;
        rc = p.transB ? copy_operand(B, ldb, N, K, true, stream, &bscratch, &pitch, pre_b)
                      : copy_operand(B, ldb, K, N, false, stream, &bscratch, &pitch, pre_b);
        if (rc != REPOPS_OK) return fail(rc);
        if (bscratch) {
            p.B = static_cast<const float *>(bscratch);
            p.ldb = pitch;
            p.transB = 0;
            p.span_b[0] = reinterpret_cast<uintptr_t>(bscratch);
            p.span_b[1] = p.span_b[0] + uint64_t(K) * uint64_t(pitch) * 4u;
        }
    }
    if (copy_a) {
        // a K-inner A (M x K) is transposed, an unaligned M-inner A (K x M) repacked
        int64_t pitch = 0;
        rc = p.transA ? copy_operand(A, lda, K, M, false, stream, &ascratch, &pitch, pre_a)
                      : copy_operand(A, lda, M, K, true, stream, &ascratch, &pitch, pre_a);
        if (rc != REPOPS_OK) return fail(rc);
        if (ascratch) {
            p.A = static_cast<const float *>(ascratch);
            p.lda = pitch;
            p.transA = 1;
            p.span_a[0] = reinterpret_cast<uintptr_t>(ascratch);
            p.span_a[1] = p.span_a[0] + uint64_t(K) * uint64_t(pitch) * 4u;
        }
    }
    tma_ok = gemm_tma_eligible(p);
    const int use = (loader == REPOPS_LOADER_CPASYNC || !tma_ok) ? REPOPS_LOADER_CPASYNC : REPOPS_LOADER_TMA;
    rc = REPOPS_ERR_UNSUPPORTED;
    if (want_sk && use == REPOPS_LOADER_TMA) {
        rc = launch_chained_split(p, cfg, sk_explicit ? sk_req : 0, need_sk ? pre_sk : nullptr);
        if (rc == REPOPS_ERR_UNSUPPORTED && sk_explicit) return fail(rc);
    }
    if (rc == REPOPS_ERR_UNSUPPORTED) rc = kLaunch[cfg](p, use);
    if (rc == REPOPS_ERR_UNSUPPORTED && use == REPOPS_LOADER_TMA && loader == REPOPS_LOADER_AUTO) {
        // the encoder refused a map: run on the caller's operands with the 4-byte loader
        p.A = A; p.lda = lda; p.B = B; p.ldb = ldb;
        p.transA = transA ? 1 : 0;
        p.transB = transB ? 1 : 0;
        set_spans(p, a_bytes, b_bytes, c_bytes);
        rc = kLaunch[cfg](p, REPOPS_LOADER_CPASYNC);
    }
    for (void *m : {bscratch != pre_b ? bscratch : nullptr, ascratch != pre_a ? ascratch : nullptr}) {
        if (!m) continue;
        cudaError_t e = cudaFreeAsync(m, stream);
        if (e != cudaSuccess && rc == REPOPS_OK) rc = set_cuda_error(e);
    }
    return rc;
}

// Span in bytes of `batch` operands `stride` elements apart, each spanning
// `one` bytes.
bool batched_span(int64_t batch, int64_t stride, uint64_t one, uint64_t *bytes) {
    if (one == 0 || batch <= 1 || stride == 0) { *bytes = one; return true; }
    const uint64_t s = uint64_t(stride) * 4u;
    if (uint64_t(batch - 1) > (uint64_t(INT64_MAX) - one) / s) return false;
    *bytes = uint64_t(batch - 1) * s + one;
    return true;
}

int gemm_dispatch_batched(int config, int loader, int transA, int transB, int64_t batch, int64_t M, int64_t N,
                          int64_t K, const float *A, int64_t lda, int64_t strideA, const float *B, int64_t ldb,
                          int64_t strideB, float *C, int64_t ldc, int64_t strideC, float alpha,
                          const float *bias, int act, const float *R, int64_t ldr, int64_t strideR,
                          int64_t causal_first, int64_t k_lo, int64_t k_hi, int64_t b_group,
                          cudaStream_t stream) {
    if (batch < 0 || M < 0 || N < 0 || K < 0) return REPOPS_ERR_INVALID_ARG;
    if (causal_first < -1 || k_lo < -1 || k_hi < -1 || b_group < 1) return REPOPS_ERR_INVALID_ARG;
    if (strideA < 0 || strideB < 0 || strideC < 0 || strideR < 0) return REPOPS_ERR_INVALID_ARG;
    if (config < -1 || config >= kGemmConfigCount) return REPOPS_ERR_INVALID_ARG;
    if (loader != REPOPS_LOADER_AUTO && loader != REPOPS_LOADER_TMA && loader != REPOPS_LOADER_CPASYNC)
        return REPOPS_ERR_INVALID_ARG;
    if (act != REPOPS_ACT_NONE && act != REPOPS_ACT_GELU) return REPOPS_ERR_INVALID_ARG;
    const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;
    if (lda < std::max<int64_t>(1, a_cols) || ldb < std::max<int64_t>(1, b_cols) ||
        ldc < std::max<int64_t>(1, N) || (R && ldr < std::max<int64_t>(1, N)))
        return REPOPS_ERR_INVALID_ARG;
    if (batch == 0 || M == 0 || N == 0) return REPOPS_OK;
    if (batch > 65535) return REPOPS_ERR_UNSUPPORTED;   // one grid row per batch
    if (!C) return REPOPS_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B)) return REPOPS_ERR_INVALID_ARG;
    uint64_t a1 = 0, b1 = 0, c1 = 0, r1 = 0, a_bytes = 0, b_bytes = 0, c_bytes = 0, r_bytes = 0;
    if (!operand_span(a_rows, a_cols, lda, &a1) || !operand_span(b_rows, b_cols, ldb, &b1) ||
        !operand_span(M, N, ldc, &c1) || (R && !operand_span(M, N, ldr, &r1)))
        return REPOPS_ERR_INVALID_ARG;
    const int64_t b_mats = (batch + b_group - 1) / b_group;   // distinct B matrices read
    if (!batched_span(batch, strideA, a1, &a_bytes) || !batched_span(b_mats, strideB, b1, &b_bytes) ||
        !batched_span(batch, strideC, c1, &c_bytes) || (R && !batched_span(batch, strideR, r1, &r_bytes)))
        return REPOPS_ERR_INVALID_ARG;
    // The batches' outputs must not overlap one another: either stacked (each
    // C_b past the end of the previous one) or interleaved within one row
    // pitch (C_b = columns [b*strideC, b*strideC + N) of shared rows).
    if (batch > 1) {
        const bool stacked = uint64_t(strideC) * 4u >= c1;
        const bool interleaved = strideC >= N && (batch - 1) * strideC + N <= ldc;
        if (!stacked && !interleaved) return REPOPS_ERR_ALIAS;
    }
    if (ranges_overlap(C, c_bytes, A, a_bytes) || ranges_overlap(C, c_bytes, B, b_bytes))
        return REPOPS_ERR_ALIAS;
    if (bias && ranges_overlap(C, c_bytes, bias, uint64_t(N) * 4u)) return REPOPS_ERR_ALIAS;
    // a residual is either C itself (each element reads its own old value
    // before writing it) or disjoint from C
    const bool r_in_place = R == C && ldr == ldc && (batch == 1 || strideR == strideC);
    if (R && !r_in_place && ranges_overlap(C, c_bytes, R, r_bytes)) return REPOPS_ERR_ALIAS;

    GemmProblem p;
    p.transA = transA ? 1 : 0;
    p.transB = transB ? 1 : 0;
    p.M = M; p.N = N; p.K = K;
    p.A = A; p.lda = lda; p.B = B; p.ldb = ldb; p.C = C; p.ldc = ldc;
    p.stream = stream;
    p.ex = true;
    p.batch = batch;
    p.strideA = batch > 1 ? strideA : 0;
    p.strideB = b_mats > 1 ? strideB : 0;
    p.b_group = b_mats > 1 ? b_group : 1;
    p.strideC = batch > 1 ? strideC : 0;
    p.alpha = alpha;
    p.bias = bias;
    p.act = act;
    p.R = R;
    p.ldr = ldr;
    p.strideR = batch > 1 ? strideR : 0;
    p.causal = causal_first < N ? causal_first : -1;   // from N on, no tile lies above the boundary
    // a bound that no row reaches leaves that side open
    p.k_lo = k_lo >= 0 && k_lo < M - 1 ? k_lo : -1;
    p.k_hi = k_hi >= 0 && k_hi < K - 1 ? k_hi : -1;
    set_spans(p, a_bytes, b_bytes, c_bytes);
    int rc = status_address(&p.status);
    if (rc != REPOPS_OK) return rc;

    const bool sk_allowed = loader == REPOPS_LOADER_AUTO && config < 0 && batch == 1 && p.causal < 0 &&
                            p.k_lo < 0 && p.k_hi < 0;
    bool sk_auto = false;
    const int cfg = config >= 0 ? config
                    : (p.k_lo >= 0 || p.k_hi >= 0) ? choose_config_banded(M, N, K, batch, p.k_lo, p.k_hi)
                                                   : choose_plan(M, N, K, batch, sk_allowed, &sk_auto);
    // K == 0 has no k-slices to copy: the cp.async kernel runs the epilogue on +0
    bool tma_ok = K > 0 && gemm_tma_eligible(p);
    if (loader == REPOPS_LOADER_TMA && !tma_ok) return REPOPS_ERR_UNSUPPORTED;
    // One large product (a projection with its epilogue): a row-major A runs the
    // M-inner kernels on a transposed scratch copy, as in gemm_dispatch (3%
    // faster at 8192^3; same bits).  Batches of attention products keep their
    // layouts: their A (probabilities) would cost as much to copy as they gain.
    void *ascratch = nullptr;
    if (loader == REPOPS_LOADER_AUTO && batch == 1 && tma_ok && !p.transA &&
        2.0 * double(M) * double(N) * double(K) >= kRepackMinFlops) {
        int64_t pitch = 0;
        rc = copy_operand(A, lda, M, K, true, stream, &ascratch, &pitch);
        if (rc != REPOPS_OK) return rc;
        if (ascratch) {
            p.A = static_cast<const float *>(ascratch);
            p.lda = pitch;
            p.transA = 1;
            p.span_a[0] = reinterpret_cast<uintptr_t>(ascratch);
            p.span_a[1] = p.span_a[0] + uint64_t(K) * uint64_t(pitch) * 4u;
        }
    }
    const int use = (loader == REPOPS_LOADER_CPASYNC || !tma_ok) ? REPOPS_LOADER_CPASYNC : REPOPS_LOADER_TMA;
    rc = REPOPS_ERR_UNSUPPORTED;
    if (sk_auto && use == REPOPS_LOADER_TMA) rc = launch_chained_split(p, cfg, 0);
    if (rc == REPOPS_ERR_UNSUPPORTED) rc = kLaunch[cfg](p, use);
    if (rc == REPOPS_ERR_UNSUPPORTED && use == REPOPS_LOADER_TMA && loader == REPOPS_LOADER_AUTO) {
        p.A = A; p.lda = lda; p.transA = transA ? 1 : 0;
        set_spans(p, a_bytes, b_bytes, c_bytes);
        rc = kLaunch[cfg](p, REPOPS_LOADER_CPASYNC);   // the encoder refused a map
    }
    if (ascratch) {
        cudaError_t e = cudaFreeAsync(ascratch, stream);
        if (e != cudaSuccess && rc == REPOPS_OK) rc = set_cuda_error(e);
    }
    return rc;
}

}  // namespace

namespace gemm {
EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}
}  // namespace gemm

bool gemm_tma_eligible(const GemmProblem &p) {
    if (!gemm::tensor_map_encoder()) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p.A), b = reinterpret_cast<uintptr_t>(p.B);
    if (a % 16 || b % 16) return false;          // tensor-map base alignment
    if (p.lda % 4 || p.ldb % 4) return false;    // row pitch: multiple of 16 bytes
    if (p.lda >= (int64_t(1) << 37) || p.ldb >= (int64_t(1) << 37)) return false;   // pitch < 2^40 B
    const int64_t lim = int64_t(1) << 31;        // int32 box coordinates
    if (p.M >= lim || p.N >= lim || p.K >= lim) return false;
    if (p.ex && p.batch > 1) {
        // a batch stride is the pitch of a third map dimension: a multiple of
        // 16 bytes below 2^40 bytes (0 = shared operand, no third dimension)
        for (int64_t st : {p.strideA, p.strideB})
            if (st % 4 || st >= (int64_t(1) << 37)) return false;
    }
    return true;
}

int gemm_read_and_clear_device_status(cudaStream_t stream, unsigned *value) {
    unsigned *addr = nullptr;
    int rc = status_address(&addr);
    if (rc != REPOPS_OK) return rc;
    unsigned v = 0, zero = 0;
    cudaError_t e = cudaMemcpyAsync(&v, addr, sizeof(v), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(addr, &zero, sizeof(zero), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return set_cuda_error(e);
    *value = v;
    return REPOPS_OK;
}

}  // namespace repops

using namespace repops;

extern "C" int repops_gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                               const float *B, int64_t ldb, float *C, int64_t ldc,
                               cudaStream_t stream) {
    return gemm_dispatch(-1, REPOPS_LOADER_AUTO, 0, 0, M, N, K, A, lda, B, ldb, C, ldc, stream);
}

extern "C" uint64_t repops_gemm_workspace_bytes(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                                const float *A, int64_t lda, const float *B, int64_t ldb) {
    uint64_t need = 0;
    const int64_t ldc = std::max<int64_t>(N, 1);
    if (gemm_dispatch(-1, REPOPS_LOADER_AUTO, transA, transB, M, N, K, A, lda, B, ldb, nullptr, ldc, nullptr,
                      kSkAuto, nullptr, 0, &need) != REPOPS_OK)
        return 0;
    return need;
}

extern "C" int repops_gemm_f32_ws(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A,
                                  int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc,
                                  void *workspace, uint64_t workspace_bytes, cudaStream_t stream) {
    if (!workspace && workspace_bytes) return REPOPS_ERR_INVALID_ARG;
    return gemm_dispatch(-1, REPOPS_LOADER_AUTO, transA, transB, M, N, K, A, lda, B, ldb, C, ldc, stream,
                         kSkAuto, workspace, workspace_bytes);
}

extern "C" int repops_gemm_f32_ex(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                  const float *A, int64_t lda, const float *B, int64_t ldb, float *C,
                                  int64_t ldc, cudaStream_t stream) {
    return gemm_dispatch(-1, REPOPS_LOADER_AUTO, transA, transB, M, N, K, A, lda, B, ldb, C, ldc,
                         stream);
}

extern "C" int repops_gemm_f32_config(int config, int loader, int transA, int transB, int64_t M,
                                      int64_t N, int64_t K, const float *A, int64_t lda,
                                      const float *B, int64_t ldb, float *C, int64_t ldc,
                                      cudaStream_t stream) {
    return gemm_dispatch(config, loader, transA, transB, M, N, K, A, lda, B, ldb, C, ldc, stream);
}

extern "C" int repops_gemm_f32_chained(int config, int workers, int transA, int transB, int64_t M, int64_t N,
                                       int64_t K, const float *A, int64_t lda, const float *B, int64_t ldb,
                                       float *C, int64_t ldc, cudaStream_t stream) {
    if (workers < 0) return REPOPS_ERR_INVALID_ARG;
    return gemm_dispatch(config, REPOPS_LOADER_TMA, transA, transB, M, N, K, A, lda, B, ldb, C, ldc, stream,
                         workers);
}

extern "C" int repops_gemm_f32_batched(int config, int loader, int transA, int transB, int64_t batch,
                                       int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                       int64_t strideA, const float *B, int64_t ldb, int64_t strideB,
                                       float *C, int64_t ldc, int64_t strideC, float alpha,
                                       const float *bias, int act, const float *R, int64_t ldr,
                                       int64_t strideR, int64_t causal_first, int64_t k_lo, int64_t k_hi,
                                       int64_t b_group, cudaStream_t stream) {
    return gemm_dispatch_batched(config, loader, transA, transB, batch, M, N, K, A, lda, strideA, B, ldb,
                                 strideB, C, ldc, strideC, alpha, bias, act, R, ldr, strideR, causal_first,
                                 k_lo, k_hi, b_group, stream);
}

namespace {

// Ordered teardown of the helper streams and events of one host-buffer call:
// destruction is deferred by the runtime until their pending work completes.
struct HostCallResources {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev[4 + 2 * 64] = {};
    int nev = 0;
    ~HostCallResources() {
        for (int i = 0; i < nev; ++i)
            if (ev[i]) cudaEventDestroy(ev[i]);
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
    }
    cudaError_t event(cudaEvent_t *e) {
        cudaError_t r = cudaEventCreateWithFlags(&ev[nev], cudaEventDisableTiming);
        if (r == cudaSuccess) *e = ev[nev++];
        return r;
    }
};

}  // namespace

extern "C" int repops_gemm_f32_host(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                                    int64_t ldb, float *C, int64_t ldc, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return REPOPS_ERR_INVALID_ARG;
    if (lda < std::max<int64_t>(1, K) || ldb < std::max<int64_t>(1, N) || ldc < std::max<int64_t>(1, N))
        return REPOPS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return REPOPS_OK;
    if (!C || (K > 0 && (!A || !B))) return REPOPS_ERR_INVALID_ARG;
    uint64_t ab = 0, bb = 0, cb = 0;
    if (!operand_span(M, K, lda, &ab) || !operand_span(K, N, ldb, &bb) || !operand_span(M, N, ldc, &cb))
        return REPOPS_ERR_INVALID_ARG;
    if (ranges_overlap(C, cb, A, ab) || ranges_overlap(C, cb, B, bb)) return REPOPS_ERR_ALIAS;
    // device copies with a 16-byte pitch (the TMA loader's rule)
    const int64_t pk = std::max<int64_t>(4, (K + 3) / 4 * 4), pn = (N + 3) / 4 * 4;   // pitches >= 1 even for K = 0
    const size_t bytesA = size_t(M) * size_t(pk) * 4u, bytesB = size_t(K) * size_t(pn) * 4u;
    const size_t bytesC = size_t(M) * size_t(pn) * 4u;
    // A's row blocks: about four, each a multiple of 128 rows, at most 64
    const int64_t rows = std::max<int64_t>(128, (M / 4 + 127) / 128 * 128);
    const int blocks = int(std::min<int64_t>((M + rows - 1) / rows, 64));
    const int64_t step = (M + blocks - 1) / blocks;
    HostCallResources res;
    cudaError_t e = cudaStreamCreateWithFlags(&res.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&res.out, cudaStreamNonBlocking);
    if (e != cudaSuccess) return set_cuda_error(e);
    void *mem = nullptr;
    if (scratch_malloc(&mem, bytesA + bytesB + bytesC, stream) != cudaSuccess) {
        cudaGetLastError();
        return REPOPS_ERR_ALLOC;
    }
    float *dA = static_cast<float *>(mem), *dB = dA + bytesA / 4, *dC = dB + bytesB / 4;
    cudaEvent_t ready, b_in;
    int rc = REPOPS_OK;
    if ((e = res.event(&ready)) != cudaSuccess || (e = res.event(&b_in)) != cudaSuccess) {
        cudaFreeAsync(mem, stream);
        return set_cuda_error(e);
    }
    // the helper streams start once the allocation is ordered on `stream`
    if (rc == REPOPS_OK && ((e = cudaEventRecord(ready, stream)) != cudaSuccess ||
                            (e = cudaStreamWaitEvent(res.in, ready, 0)) != cudaSuccess ||
                            (e = cudaStreamWaitEvent(res.out, ready, 0)) != cudaSuccess))
        rc = set_cuda_error(e);
    if (rc == REPOPS_OK && K > 0 &&
        ((e = cudaMemcpy2DAsync(dB, size_t(pn) * 4u, B, size_t(ldb) * 4u, size_t(N) * 4u, size_t(K),
                                cudaMemcpyHostToDevice, res.in)) != cudaSuccess ||
         (e = cudaEventRecord(b_in, res.in)) != cudaSuccess ||
         (e = cudaStreamWaitEvent(stream, b_in, 0)) != cudaSuccess))
        rc = set_cuda_error(e);
    for (int i = 0; rc == REPOPS_OK && i < blocks; ++i) {
        const int64_t r0 = int64_t(i) * step, r1 = std::min<int64_t>(M, r0 + step);
        if (r0 >= r1) break;
        cudaEvent_t a_in, c_done;
        if ((e = res.event(&a_in)) != cudaSuccess || (e = res.event(&c_done)) != cudaSuccess) {
            rc = set_cuda_error(e);
            break;
        }
        if (K > 0 && ((e = cudaMemcpy2DAsync(dA + r0 * pk, size_t(pk) * 4u, A + r0 * lda, size_t(lda) * 4u,
                                             size_t(K) * 4u, size_t(r1 - r0), cudaMemcpyHostToDevice, res.in)) !=
                          cudaSuccess ||
                      (e = cudaEventRecord(a_in, res.in)) != cudaSuccess ||
                      (e = cudaStreamWaitEvent(stream, a_in, 0)) != cudaSuccess)) {
            rc = set_cuda_error(e);
            break;
        }
        rc = gemm_dispatch(-1, REPOPS_LOADER_AUTO, 0, 0, r1 - r0, N, K, dA + r0 * pk, pk, dB, pn, dC + r0 * pn, pn,
                           stream);
        if (rc != REPOPS_OK) break;
        if ((e = cudaEventRecord(c_done, stream)) != cudaSuccess || (e = cudaStreamWaitEvent(res.out, c_done, 0)) != cudaSuccess ||
            (e = cudaMemcpy2DAsync(C + r0 * ldc, size_t(ldc) * 4u, dC + r0 * pn, size_t(pn) * 4u, size_t(N) * 4u,
                                   size_t(r1 - r0), cudaMemcpyDeviceToHost, res.out)) != cudaSuccess)
            rc = set_cuda_error(e);
    }
    // `stream` resumes after every copy in and back (or what an error left
    // queued); then the memory is released
    if ((e = join_helper_streams(stream, res.in, res.out)) != cudaSuccess && rc == REPOPS_OK) rc = set_cuda_error(e);
    e = cudaFreeAsync(mem, stream);
    if (rc == REPOPS_OK && e != cudaSuccess) rc = set_cuda_error(e);
    return rc;
}

extern "C" int repops_gemm_config_count(void) { return kGemmConfigCount; }

extern "C" int repops_gemm_small_output(int64_t M, int64_t N, int64_t K) { return repops::small_output(M, N, K) ? 1 : 0; }

extern "C" int repops_gemm_config_info(int config, int *bm, int *bn, int *threads, int *tm, int *tn) {
    if (config < 0 || config >= kGemmConfigCount) return REPOPS_ERR_INVALID_ARG;
    const GemmConfigInfo ci = config_info(config);
    if (bm) *bm = ci.bm;
    if (bn) *bn = ci.bn;
    if (threads) *threads = ci.threads;
    if (tm) *tm = ci.tm;
    if (tn) *tn = ci.tn;
    return REPOPS_OK;
}

extern "C" int repops_gemm_config_occupancy(int config) {
    if (config < 0 || config >= kGemmConfigCount) return REPOPS_ERR_INVALID_ARG;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != REPOPS_OK) return rc;
    if (di.device < 0 || di.device >= kMaxDevices) return REPOPS_ERR_UNSUPPORTED;
    return occupancy_of(di.device, config);
}

extern "C" int repops_gemm_auto_config(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0) return -1;
    return choose_plan(M, N, std::max<int64_t>(K, 1), 1, true, nullptr);
}

extern "C" int repops_gemm_auto_chained(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || small_output(M, N, K)) return 0;
    bool sk = false;
    choose_plan(M, N, K, 1, true, &sk);
    return sk ? 1 : 0;
}

extern "C" int repops_set_thread_status_word(unsigned *word) {
    if (reinterpret_cast<uintptr_t>(word) % 4) return REPOPS_ERR_INVALID_ARG;
    t_status_word = word;
    return REPOPS_OK;
}

extern "C" int repops_selftest_bounded_wait(int64_t limit_ns, cudaStream_t stream) {
    if (limit_ns < 1 || limit_ns > int64_t(kWaitLimitNs)) return REPOPS_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    int rc = status_address(&status);
    if (rc != REPOPS_OK) return rc;
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(status, uint64_t(limit_ns));
    return check_launch();
}

extern "C" int repops_selftest_bounded_flag_wait(int64_t limit_ns, cudaStream_t stream) {
    if (limit_ns < 1 || limit_ns > int64_t(kWaitLimitNs)) return REPOPS_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    int rc = status_address(&status);
    if (rc != REPOPS_OK) return rc;
    flag_wait_selftest_kernel<<<1, 32, 0, stream>>>(status, uint64_t(limit_ns));
    return check_launch();
}
