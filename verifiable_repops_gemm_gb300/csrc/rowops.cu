// rowops.cu -- order-fixed row operators: softmax, LayerNorm, RMSNorm, GeLU.
//
// "Verde与RepOps" §3.2: dimensions whose order matters run serially or with
// synchronised threads; §3.3 and §4.3: LayerNorm, GeLU and ERF are the
// operators behind DistilBERT's overhead.  The pages fix no algorithm for
// them, so the library defines one whose every operation is a single IEEE
// binary32 rounding in a fixed order -- the same bits on any hardware:
//   - a reduction over a row is a fixed 32-ary tree: each run of 32
//     consecutive values is folded left to right from its first value, the run
//     results are folded the same way, level by level, until one value is left
//     (max keeps the earlier value unless a later one is strictly greater);
//   - exp(x): k = rint(x * log2 e); r = (x - k*ln2_hi) - k*ln2_lo (Cody and
//     Waite's two-part ln 2, k*ln2_hi exact); e^r by the degree-7 Taylor
//     polynomial in Horner form; times 2^k by exact power-of-two scaling;
//   - erfc(z), z >= 0: the Chebyshev fit of Numerical Recipes §6.2 (Press,
//     Teukolsky, Vetterling, Flannery), with the exp above;
//   - GeLU(x) = 0.5*x*(1 + erf(x/sqrt 2)) with 1 + erf(z) = 2 - erfc(z) for
//     z >= 0 and erfc(-z) for z < 0;
//   - a row's normaliser is one correctly rounded reciprocal per row (1/s for
//     softmax, 1/sqrt(var + eps) for the norms: __frcp_rn of __fsqrt_rn),
//     applied to each element by one multiplication; products and sums never
//     fuse.
//
// Kernels: one CTA per row, persistent over rows.  Each thread owns whole runs
// (R runs of 32 values, in registers) and folds them; a warp folds its 32 run
// results by shuffles, and the group results meet in shared memory after one
// barrier per reduction; the row is read once and written once.  Aligned rows move between HBM and registers through a
// shared-memory stage: each warp copies its 32 consecutive runs (4 KB) with
// coalesced 16-byte cp.async, each lane then reads its own run; the next row's
// copy is in flight while the current row is reduced.  Outputs leave the same
// way.  Rows longer than 32 * 256 * 4 values, and rows that are not 16-byte
// aligned, use a kernel that re-reads the row for each phase.
#include <algorithm>

#include "fixed_math.cuh"
#include "internal.cuh"

namespace repops {
namespace {

constexpr int RUN = 32;

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
constexpr int MAX_FAST_RUNS = 256 * 4;          // register-resident rows: up to 32768 values
constexpr int MAX_GENERIC_RUNS = 12288;         // run results in 48 KB of shared memory

// Resident CTAs per SM the staged backward kernels ask the compiler for.
// Softmax backward: 10 warps (about 100 registers a thread for its p and dp
// runs), measured 11% faster than the uncapped 151 registers; the forward
// softmax kernels stay uncapped (capped at 64 registers they ran 13% slower:
// their 32 exponentials a thread need the registers for overlap).
template <int T>
constexpr int kBwdRowBlocks = T == 32 ? 16 : 640 / T;
// RMSNorm backward: 16 warps (128 registers; x, dy, gamma and res runs live).
template <int T>
constexpr int kNormBwdBlocks = T == 32 ? 12 : 512 / T;

// ------------------------------------------------------------ arithmetic ----

enum class Op { Sum, Max };

template <Op OP>
__device__ __forceinline__ float combine(float acc, float v) {
    if constexpr (OP == Op::Sum) return __fadd_rn(acc, v);
    else return v > acc ? v : acc;
}

// Upper levels of the tree over the m run results in a[] (shared memory),
// ping-ponging with b[]; every thread of the CTA calls it and receives the
// root.  Both buffers are clobbered.
template <Op OP>
__device__ float tree_upper(float *a, float *b, int m, float *bcast) {
    __syncthreads();
    while (m > 1) {
        const int groups = (m + RUN - 1) / RUN;
        for (int g = threadIdx.x; g < groups; g += blockDim.x) {
            const int s = g * RUN, e = min(s + RUN, m);
            float acc = a[s];
            for (int i = s + 1; i < e; ++i) acc = combine<OP>(acc, a[i]);
            b[g] = acc;
        }
        __syncthreads();
        float *t = a; a = b; b = t;
        m = groups;
    }
    if (threadIdx.x == 0) *bcast = a[0];
    __syncthreads();
    const float r = *bcast;
    __syncthreads();
    return r;
}

// ------------------------------------------------------ register rows ----

// A thread's R runs of one row: run j of the thread is run (threadIdx.x + j*T)
// of the row.  Elements past the row end are never read or written.
template <int T, int R>
struct RowRuns {
    float v[R][RUN];
    int len[R];   // values in each run (0 when the run is past the end)

    // The tree's root over the row, to every thread.  Each thread folds its
    // runs (of f(value)) left to right; a group of 32 consecutive runs is one
    // warp's lanes for one j, and every lane folds the group's run results left
    // to right by shuffles; lane 0 posts the group result and, after one
    // barrier, every thread folds the (at most 32) group results left to right.
    // gbuf: two halves of 32 floats, alternated through `phase`, so that a
    // thread still reading one reduction's half never races the next one's
    // writes.
    template <Op OP, class F>
    __device__ __forceinline__ float reduce(F f, float (*gbuf)[RUN], int &phase, int runs) const {
        constexpr int GROUPS = T * R / RUN;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        float *gb = gbuf[phase];
        phase ^= 1;
        float root = 0.0f;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int u0 = j * T + warp * RUN;   // the group's first run
            if (u0 >= runs) continue;           // warp-uniform
            // a lane past the row end folds garbage that the group fold skips
            float acc = f(v[j][0]);
            if (len[j] == RUN) {
#pragma unroll
                for (int i = 1; i < RUN; ++i) acc = combine<OP>(acc, f(v[j][i]));
            } else {
#pragma unroll
                for (int i = 1; i < RUN; ++i)
                    if (i < len[j]) acc = combine<OP>(acc, f(v[j][i]));
            }
            const int have = runs - u0;         // runs present in the group, >= 1
            float g = __shfl_sync(0xffffffffu, acc, 0);
            if (have >= RUN) {                  // a full group (warp-uniform): no per-lane test
#pragma unroll
                for (int i = 1; i < RUN; ++i) g = combine<OP>(g, __shfl_sync(0xffffffffu, acc, i));
            } else {
#pragma unroll
                for (int i = 1; i < RUN; ++i) {
                    const float o = __shfl_sync(0xffffffffu, acc, i);
                    if (i < have) g = combine<OP>(g, o);
                }
            }
            if constexpr (GROUPS == 1) root = g;
            else if (lane == 0) gb[j * (T / RUN) + warp] = g;
        }
        if constexpr (GROUPS == 1) {
            return root;
        } else {
            __syncthreads();
            const int G = (runs + RUN - 1) / RUN;
            float r = gb[0];
            for (int k = 1; k < G; ++k) r = combine<OP>(r, gb[k]);
            return r;
        }
    }
};

// The 32 values of run `s` of a per-column vector (gamma, beta): all loads in
// flight together instead of one per element.
__device__ __forceinline__ void load_run(const float *__restrict__ p, int64_t s, int len, bool vec,
                                         float (&out)[RUN]) {
    if (vec && len == RUN) {
        const float4 *q = reinterpret_cast<const float4 *>(p + s);
#pragma unroll
        for (int k = 0; k < RUN / 4; ++k) {
            const float4 w = __ldg(q + k);
            out[4 * k] = w.x; out[4 * k + 1] = w.y; out[4 * k + 2] = w.z; out[4 * k + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < RUN; ++i) out[i] = i < len ? __ldg(p + s + i) : 0.0f;
    }
}

// ------------------------------------------------ shared-memory stage ----

// Run u of a row occupies 128 bytes of the stage at u*128; its 16-byte chunk c
// sits in slot c ^ (u & 7).  Eight consecutive lanes then hit eight different
// bank groups both when they copy eight consecutive chunks of one run and when
// each reads the same chunk of its own run.
__device__ __forceinline__ int stage_slot(int u, int c) { return u * 8 + (c ^ (u & 7)); }

// Starts the copy of the row's runs [0, T*R) into the stage; each warp copies
// the runs its own lanes own (so only __syncwarp is needed before reading).
template <int T, int R>
__device__ __forceinline__ void stage_in(float4 *stage, const float *__restrict__ row, int64_t n) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int u0 = j * T + warp * 32;
        if (int64_t(u0) * RUN >= n) continue;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int g = k * 32 + lane, u = u0 + (g >> 3), c = g & 7;
            const int64_t f = int64_t(u) * RUN + 4 * c;
            if (f < n) cp_async_16(stage + stage_slot(u, c), row + f, uint32_t(imin64(4, n - f)) * 4u);
        }
    }
}

// Stores the row's first n values from the stage with coalesced 16-byte stores.
template <int T, int R>
__device__ __forceinline__ void stage_out(const float4 *stage, float *__restrict__ row, int64_t n) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int u0 = j * T + warp * 32;
        if (int64_t(u0) * RUN >= n) continue;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int g = k * 32 + lane, u = u0 + (g >> 3), c = g & 7;
            const int64_t f = int64_t(u) * RUN + 4 * c;
            if (f >= n) continue;
            const float4 w = stage[stage_slot(u, c)];
            if (f + 4 <= n) {
                __stcs(reinterpret_cast<float4 *>(row + f), w);
            } else {
                row[f] = w.x;
                if (f + 1 < n) row[f + 1] = w.y;
                if (f + 2 < n) row[f + 2] = w.z;
            }
        }
    }
}

template <int T, int R>
__device__ __forceinline__ void read_stage(RowRuns<T, R> &rr, const float4 *stage, int64_t n) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int u = threadIdx.x + j * T;
        const int64_t s = int64_t(u) * RUN;
        rr.len[j] = s < n ? int(imin64(RUN, n - s)) : 0;
        if (rr.len[j] == 0) continue;
#pragma unroll
        for (int c = 0; c < RUN / 4; ++c) {
            const float4 w = stage[stage_slot(u, c)];
            rr.v[j][4 * c] = w.x; rr.v[j][4 * c + 1] = w.y; rr.v[j][4 * c + 2] = w.z; rr.v[j][4 * c + 3] = w.w;
        }
    }
}

template <int T, int R>
__device__ __forceinline__ void write_stage(const RowRuns<T, R> &rr, float4 *stage) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
        if (rr.len[j] == 0) continue;
        const int u = threadIdx.x + j * T;
#pragma unroll
        for (int c = 0; c < RUN / 4; ++c)
            stage[stage_slot(u, c)] =
                make_float4(rr.v[j][4 * c], rr.v[j][4 * c + 1], rr.v[j][4 * c + 2], rr.v[j][4 * c + 3]);
    }
}

// A per-column vector (gamma, beta) staged once per CTA in the same layout,
// read back one run at a time.
template <int T, int R>
__device__ __forceinline__ void read_param_run(const float4 *pstage, int u, float (&out)[RUN]) {
#pragma unroll
    for (int c = 0; c < RUN / 4; ++c) {
        const float4 w = pstage[stage_slot(u, c)];
        out[4 * c] = w.x; out[4 * c + 1] = w.y; out[4 * c + 2] = w.z; out[4 * c + 3] = w.w;
    }
}

// Two stages (the next row's copy overlaps this row's work) while they fit in
// 128 KB; one beyond.
template <int T, int R>
constexpr bool kPrefetch = T * R <= 512;
template <int T, int R>
constexpr size_t kStageBytes = size_t(T) * R * RUN * sizeof(float) * (kPrefetch<T, R> ? 2 : 1);
// NP per-column vectors staged after the row stages when all fit in 200 KB.
template <int T, int R, int NP>
constexpr size_t kParamBytes =
    kStageBytes<T, R> + size_t(NP) * T * R * RUN * sizeof(float) <= 200 * 1024 ? size_t(NP) * T * R * RUN * 4 : 0;

// The row loop shared by the three row kernels: body(rr, row) turns the row's
// values in rr into its outputs.  x, y and their leading dimensions are
// 16-byte aligned (other rows take the long-row kernel).
template <int T, int R, class Body>
__device__ __forceinline__ void for_each_row(int64_t rows, int64_t n, const float *__restrict__ x, int64_t ldx,
                                             float *__restrict__ y, int64_t ldy, Body body) {
    extern __shared__ float4 stage_mem[];
    constexpr bool PF = kPrefetch<T, R>;
    float4 *in = stage_mem;
    float4 *out = PF ? stage_mem + T * R * RUN / 4 : stage_mem;
    int64_t row = blockIdx.x;
    if (row < rows) stage_in<T, R>(in, x + row * ldx, n);
    cp_async_commit();
    for (; row < rows; row += gridDim.x) {
        const int64_t next = row + gridDim.x;
        cp_async_wait<0>();
        __syncwarp();
        RowRuns<T, R> rr;
        read_stage(rr, in, n);
        if constexpr (PF) {
            __syncwarp();                       // every lane has its run before `in` is refilled
            if (next < rows) stage_in<T, R>(in, x + next * ldx, n);
            cp_async_commit();
        }
        body(rr, row);
        write_stage(rr, out);
        __syncwarp();
        stage_out<T, R>(out, y + row * ldy, n);
        __syncwarp();                           // `out` read back before it is written again
        if constexpr (!PF) {
            if (next < rows) stage_in<T, R>(in, x + next * ldx, n);
            cp_async_commit();
        }
    }
    cp_async_wait<0>();
}

// (a, b) <- (exp(a - m), exp(b - m)), the subtractions as one packed add of -m
__device__ __forceinline__ void exp_minus2(float &a, float &b, float m) {
    float d0, d1;
    unpack2(add2_rn(pack2(a, b), pack2(-m, -m)), d0, d1);
    const float2 e = exp_fixed2(d0, d1);
    a = e.x;
    b = e.y;
}

struct Ident {
    __device__ __forceinline__ float operator()(float x) const { return x; }
};
struct Square {
    __device__ __forceinline__ float operator()(float x) const { return __fmul_rn(x, x); }
};

template <int T, int R>
__global__ void __launch_bounds__(T)
softmax_rows_kernel(int64_t rows, int64_t n, const float *__restrict__ x, int64_t ldx, float *__restrict__ y,
                    int64_t ldy) {
    __shared__ float gbuf[2][RUN];
    int phase = 0;
    const int runs = int((n + RUN - 1) / RUN);
    for_each_row<T, R>(rows, n, x, ldx, y, ldy, [&](RowRuns<T, R> &rr, int64_t) {
        const float m = rr.template reduce<Op::Max>(Ident(), gbuf, phase, runs);
        // element-wise steps need no guard: values past the row end are never
        // folded or stored
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int i = 0; i < RUN; i += 2) exp_minus2(rr.v[j][i], rr.v[j][i + 1], m);
        const float inv = __frcp_rn(rr.template reduce<Op::Sum>(Ident(), gbuf, phase, runs));
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int i = 0; i < RUN; ++i) rr.v[j][i] = __fmul_rn(rr.v[j][i], inv);
    });
}

// Causal softmax: row r is the softmax of its prefix of L = min(n, first +
// (r mod period) + 1) values (the max and sum trees over those L values), then
// +0.  Only the prefix is copied in and only its exponentials are computed;
// the row loop is for_each_row's with the copy-in cut at L.
template <int T, int R>
__global__ void __launch_bounds__(T)
softmax_causal_rows_kernel(int64_t rows, int64_t n, const float *__restrict__ x, int64_t ldx,
                           float *__restrict__ y, int64_t ldy, int64_t first, int64_t period) {
    extern __shared__ float4 stage_mem[];
    __shared__ float gbuf[2][RUN];
    int phase = 0;
    constexpr bool PF = kPrefetch<T, R>;
    float4 *in = stage_mem;
    float4 *out = PF ? stage_mem + T * R * RUN / 4 : stage_mem;
    auto prefix = [&](int64_t r) { return imin64(n, first + r % period + 1); };
    int64_t row = blockIdx.x;
    if (row < rows) stage_in<T, R>(in, x + row * ldx, prefix(row));
    cp_async_commit();
    for (; row < rows; row += gridDim.x) {
        const int64_t next = row + gridDim.x;
        const int64_t L = prefix(row);
        cp_async_wait<0>();
        __syncwarp();
        RowRuns<T, R> rr;
        read_stage(rr, in, L);
        if constexpr (PF) {
            __syncwarp();                       // every lane has its run before `in` is refilled
            if (next < rows) stage_in<T, R>(in, x + next * ldx, prefix(next));
            cp_async_commit();
        }
        const int runs = int((L + RUN - 1) / RUN);
        const float m = rr.template reduce<Op::Max>(Ident(), gbuf, phase, runs);
#pragma unroll
        for (int j = 0; j < R; ++j) {
            // runs past the prefix are skipped whole; inside a run every value
            // is exponentiated (branch-free; the ones past the prefix are
            // neither folded nor stored)
            if (rr.len[j] == 0) continue;
#pragma unroll
            for (int i = 0; i < RUN; i += 2) exp_minus2(rr.v[j][i], rr.v[j][i + 1], m);
        }
        const float inv = __frcp_rn(rr.template reduce<Op::Sum>(Ident(), gbuf, phase, runs));
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int64_t s0 = int64_t(threadIdx.x + j * T) * RUN;
#pragma unroll
            for (int i = 0; i < RUN; ++i) rr.v[j][i] = i < rr.len[j] ? __fmul_rn(rr.v[j][i], inv) : 0.0f;
            rr.len[j] = s0 < n ? int(imin64(RUN, n - s0)) : 0;      // the whole row is written
        }
        write_stage(rr, out);
        __syncwarp();
        stage_out<T, R>(out, y + row * ldy, n);
        __syncwarp();                           // `out` read back before it is written again
        if constexpr (!PF) {
            if (next < rows) stage_in<T, R>(in, x + next * ldx, prefix(next));
            cp_async_commit();
        }
    }
    cp_async_wait<0>();
}

// Causal softmax with one warp per row and no CTA-wide barrier, for aligned
// rows of at most WARP_CAUSAL_MAX_COLS values: a short prefix no longer keeps
// a whole CTA waiting at the row's barriers.  The warp copies the prefix into
// its own shared-memory row (16-byte groups of each 32-value run permuted by
// the run index, so that a lane per run reads without bank conflicts and
// 4 consecutive values stay contiguous), folds the max tree (a lane per run,
// then shuffles), exponentiates with every lane (4 values at a time, in
// place), folds the sum tree the same way, and writes the row: e * (1/s) in
// the prefix, +0 after.  The same operations as softmax_causal_rows_kernel.
constexpr int WARP_CAUSAL_MAX_COLS = 4096;
constexpr int WARP_CAUSAL_WARPS = 4;

__device__ __forceinline__ int wc_pos(int j) { return (j & ~31) | ((j & 31) ^ (((j >> 5) & 7) << 2)); }

// Run results of a row held by lane l for runs l, l + 32, l + 64, l + 96
// (present below nruns): the tree's upper levels, to every lane.
template <Op OP>
__device__ __forceinline__ float warp_runs_root(const float (&rr)[4], int nruns) {
    float root = 0.0f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int have = nruns - 32 * g;
        if (have <= 0) break;                       // warp-uniform
        float acc = __shfl_sync(0xffffffffu, rr[g], 0);
#pragma unroll
        for (int i = 1; i < 32; ++i) {
            const float o = __shfl_sync(0xffffffffu, rr[g], i);
            if (i < have) acc = combine<OP>(acc, o);
        }
        root = g == 0 ? acc : combine<OP>(root, acc);
    }
    return root;
}

// The fold of one 32-value run of a staged row, left to right over its first
// len values.
template <Op OP>
__device__ __forceinline__ float fold_run(const float *run, int u, int len) {
    float acc = 0.0f;
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
        const float4 t = *reinterpret_cast<const float4 *>(run + 4 * (q4 ^ (u & 7)));
        const float v4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = 4 * q4 + e;
            if (idx == 0) acc = v4[0];
            else if (idx < len) acc = combine<OP>(acc, v4[e]);
        }
    }
    return acc;
}

__global__ void __launch_bounds__(32 * WARP_CAUSAL_WARPS)
softmax_causal_warp_kernel(int64_t rows, int n, const float *__restrict__ x, int64_t ldx, float *__restrict__ y,
                           int64_t ldy, int64_t first, int64_t period, int row_floats, unsigned *status) {
    extern __shared__ float4 wc_smem4[];
    if (!REPOPS_DBG_SMEM_OK(uint64_t(WARP_CAUSAL_WARPS) * row_floats * sizeof(float), status)) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float *stage = reinterpret_cast<float *>(wc_smem4) + warp * row_floats;
    const int64_t gw = int64_t(blockIdx.x) * WARP_CAUSAL_WARPS + warp;
    const int64_t nw = int64_t(gridDim.x) * WARP_CAUSAL_WARPS;
    for (int64_t row = gw; row < rows; row += nw) {
        const int L = int(imin64(n, first + row % period + 1));
        const float *xr = x + row * ldx;
        // the prefix, 16 bytes a copy (a short last group reads only its values)
        for (int j4 = 4 * lane; j4 < L; j4 += 128) {
            const int have = L - j4;
            cp_async_16(stage + wc_pos(j4), xr + j4, have >= 4 ? 16u : uint32_t(have) * 4u);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncwarp();
        const int nruns = (L + RUN - 1) / RUN;
        float rr[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int u = lane + 32 * g;
            rr[g] = u < nruns ? fold_run<Op::Max>(stage + 32 * u, u, min(RUN, L - 32 * u)) : 0.0f;
        }
        const float m = warp_runs_root<Op::Max>(rr, nruns);
        __syncwarp();                               // every run read before it is overwritten
        for (int j4 = 4 * lane; j4 < L; j4 += 128) {
            float4 *p4 = reinterpret_cast<float4 *>(stage + wc_pos(j4));
            float4 t = *p4;
            exp_minus2(t.x, t.y, m);
            exp_minus2(t.z, t.w, m);
            *p4 = t;
        }
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int u = lane + 32 * g;
            rr[g] = u < nruns ? fold_run<Op::Sum>(stage + 32 * u, u, min(RUN, L - 32 * u)) : 0.0f;
        }
        const float inv = __frcp_rn(warp_runs_root<Op::Sum>(rr, nruns));
        float *yr = y + row * ldy;
        for (int j4 = 4 * lane; j4 < n; j4 += 128) {
            float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (j4 < L) {
                t = *reinterpret_cast<const float4 *>(stage + wc_pos(j4));
                t.x = j4 + 0 < L ? __fmul_rn(t.x, inv) : 0.0f;
                t.y = j4 + 1 < L ? __fmul_rn(t.y, inv) : 0.0f;
                t.z = j4 + 2 < L ? __fmul_rn(t.z, inv) : 0.0f;
                t.w = j4 + 3 < L ? __fmul_rn(t.w, inv) : 0.0f;
            }
            if (j4 + 3 < n) {
                __stcs(reinterpret_cast<float4 *>(yr + j4), t);
            } else {                                // the row's last, short group
                const float v[4] = {t.x, t.y, t.z, t.w};
                for (int e = 0; j4 + e < n; ++e) yr[j4 + e] = v[e];
            }
        }
        __syncwarp();                               // the stage is refilled by the next row
    }
}

// psm: gamma and beta are staged in shared memory (aligned, and they fit).
template <int T, int R>
__global__ void __launch_bounds__(T)
layernorm_rows_kernel(int64_t rows, int64_t n, const float *__restrict__ x, int64_t ldx,
                      const float *__restrict__ gamma, const float *__restrict__ beta, float eps,
                      float *__restrict__ y, int64_t ldy, int pvec, int psm) {
    extern __shared__ float4 stage_mem[];
    __shared__ float gbuf[2][RUN];
    int phase = 0;
    const int runs = int((n + RUN - 1) / RUN);
    const float nf = float(n);
    float4 *pg = stage_mem + kStageBytes<T, R> / 16, *pb = pg + T * R * RUN / 4;
    if (kParamBytes<T, R, 2> != 0 && psm && blockIdx.x < rows) {
        stage_in<T, R>(pg, gamma, n);   // waited for with the first row
        stage_in<T, R>(pb, beta, n);
    }
    for_each_row<T, R>(rows, n, x, ldx, y, ldy, [&](RowRuns<T, R> &rr, int64_t) {
        const float mean = __fdiv_rn(rr.template reduce<Op::Sum>(Ident(), gbuf, phase, runs), nf);
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int i = 0; i < RUN; ++i) rr.v[j][i] = __fsub_rn(rr.v[j][i], mean);
        const float var = __fdiv_rn(rr.template reduce<Op::Sum>(Square(), gbuf, phase, runs), nf);
        const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(var, eps)));
#pragma unroll
        for (int j = 0; j < R; ++j) {
            if (rr.len[j] == 0) continue;
            const int u = threadIdx.x + j * T;
            float g[RUN], b[RUN];
            if (kParamBytes<T, R, 2> != 0 && psm) {
                read_param_run<T, R>(pg, u, g);
                read_param_run<T, R>(pb, u, b);
            } else {
                load_run(gamma, int64_t(u) * RUN, rr.len[j], pvec, g);
                load_run(beta, int64_t(u) * RUN, rr.len[j], pvec, b);
            }
#pragma unroll
            for (int i = 0; i < RUN; ++i) rr.v[j][i] = __fadd_rn(__fmul_rn(__fmul_rn(rr.v[j][i], inv), g[i]), b[i]);
        }
    });
}

template <int T, int R>
__global__ void __launch_bounds__(T)
rmsnorm_rows_kernel(int64_t rows, int64_t n, const float *__restrict__ x, int64_t ldx,
                    const float *__restrict__ gamma, float eps, float *__restrict__ y, int64_t ldy, int pvec,
                    int psm) {
    extern __shared__ float4 stage_mem[];
    __shared__ float gbuf[2][RUN];
    int phase = 0;
    const int runs = int((n + RUN - 1) / RUN);
    const float nf = float(n);
    float4 *pg = stage_mem + kStageBytes<T, R> / 16;
    if (kParamBytes<T, R, 1> != 0 && psm && blockIdx.x < rows) stage_in<T, R>(pg, gamma, n);
    for_each_row<T, R>(rows, n, x, ldx, y, ldy, [&](RowRuns<T, R> &rr, int64_t) {
        const float ms = __fdiv_rn(rr.template reduce<Op::Sum>(Square(), gbuf, phase, runs), nf);
        const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
#pragma unroll
        for (int j = 0; j < R; ++j) {
            if (rr.len[j] == 0) continue;
            const int u = threadIdx.x + j * T;
            float g[RUN];
            if (kParamBytes<T, R, 1> != 0 && psm) read_param_run<T, R>(pg, u, g);
            else load_run(gamma, int64_t(u) * RUN, rr.len[j], pvec, g);
#pragma unroll
            for (int i = 0; i < RUN; ++i) rr.v[j][i] = __fmul_rn(__fmul_rn(rr.v[j][i], inv), g[i]);
        }
    });
}

// ------------------------------------------------------ long rows ----

// Run results of f over the row, each run folded from global memory.
template <Op OP, class F>
__device__ float generic_reduce(const float *__restrict__ row, int64_t n, F f, float *buf, float *buf2,
                                float *bcast) {
    const int runs = int((n + RUN - 1) / RUN);
    for (int j = threadIdx.x; j < runs; j += blockDim.x) {
        const int64_t s = int64_t(j) * RUN, e = imin64(s + RUN, n);
        float acc = f(row[s]);
        for (int64_t i = s + 1; i < e; ++i) acc = combine<OP>(acc, f(row[i]));
        buf[j] = acc;
    }
    return tree_upper<OP>(buf, buf2, runs, bcast);
}

struct ExpShift {
    float m;
    __device__ __forceinline__ float operator()(float x) const { return exp_fixed(__fsub_rn(x, m)); }
};
struct SquareShift {
    float m;
    __device__ __forceinline__ float operator()(float x) const {
        const float d = __fsub_rn(x, m);
        return __fmul_rn(d, d);
    }
};

// kind 0 = softmax, 1 = LayerNorm, 2 = RMSNorm.  Each thread writes only the
// runs it read in the same pass, so y may be x.  first >= 0: causal softmax,
// row r over its first min(n, first + (r mod period) + 1) values, +0 after.
__global__ void __launch_bounds__(256)
rows_generic_kernel(int kind, int64_t rows, int64_t n, const float *__restrict__ x, int64_t ldx,
                    const float *__restrict__ gamma, const float *__restrict__ beta, float eps,
                    float *__restrict__ y, int64_t ldy, int64_t first, int64_t period, unsigned *status) {
    extern __shared__ float buf[];   // runs + ceil(runs / 32) floats
    __shared__ float bcast;
    const int runs = int((n + RUN - 1) / RUN);
    if (!REPOPS_DBG_SMEM_OK(uint64_t(runs + (runs + RUN - 1) / RUN) * sizeof(float), status)) return;
    float *buf2 = buf + runs;
    const float nf = float(n);
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *row = x + r * ldx;
        float *out = y + r * ldy;
        if (kind == 0) {
            const int64_t L = first >= 0 ? imin64(n, first + r % period + 1) : n;
            const float m = generic_reduce<Op::Max>(row, L, Ident(), buf, buf2, &bcast);
            const float inv = __frcp_rn(generic_reduce<Op::Sum>(row, L, ExpShift{m}, buf, buf2, &bcast));
            for (int j = threadIdx.x; j < runs; j += blockDim.x)
                for (int64_t i = int64_t(j) * RUN; i < imin64(int64_t(j + 1) * RUN, n); ++i)
                    out[i] = i < L ? __fmul_rn(exp_fixed(__fsub_rn(row[i], m)), inv) : 0.0f;
        } else if (kind == 1) {
            const float mean = __fdiv_rn(generic_reduce<Op::Sum>(row, n, Ident(), buf, buf2, &bcast), nf);
            const float var = __fdiv_rn(generic_reduce<Op::Sum>(row, n, SquareShift{mean}, buf, buf2, &bcast), nf);
            const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(var, eps)));
            for (int j = threadIdx.x; j < runs; j += blockDim.x)
                for (int64_t i = int64_t(j) * RUN; i < imin64(int64_t(j + 1) * RUN, n); ++i)
                    out[i] = __fadd_rn(__fmul_rn(__fmul_rn(__fsub_rn(row[i], mean), inv), gamma[i]), beta[i]);
        } else {
            const float ms = __fdiv_rn(generic_reduce<Op::Sum>(row, n, Square(), buf, buf2, &bcast), nf);
            const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
            for (int j = threadIdx.x; j < runs; j += blockDim.x)
                for (int64_t i = int64_t(j) * RUN; i < imin64(int64_t(j + 1) * RUN, n); ++i)
                    out[i] = __fmul_rn(__fmul_rn(row[i], inv), gamma[i]);
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256)
gelu_kernel(int64_t n, const float *__restrict__ x, float *__restrict__ y, int vec) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const int64_t first = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    if (vec) {
        const int64_t n4 = n / 4;
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        float4 *y4 = reinterpret_cast<float4 *>(y);
        // one float4 group a trip, the next trip's group loaded before this
        // trip's four GeLUs run
        int64_t i = first;
        const float4 zero = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        float4 v = i < n4 ? __ldcs(x4 + i) : zero;
        for (; i < n4; i += stride) {
            const bool next = i + stride < n4;
            const float4 nv = next ? __ldcs(x4 + i + stride) : zero;
            const float2 a = gelu_fixed2(v.x, v.y), b = gelu_fixed2(v.z, v.w);
            __stcs(y4 + i, make_float4(a.x, a.y, b.x, b.y));
            v = nv;
        }
        for (int64_t i = n4 * 4 + first; i < n; i += stride) y[i] = gelu_fixed(x[i]);
    } else {
        for (int64_t i = first; i < n; i += stride) y[i] = gelu_fixed(x[i]);
    }
}

// ---------------------------------------------------------- backward ----
// Backward operators of a training step, with the forward's tree and
// arithmetic: GeLU backward (element-wise), RMSNorm and softmax backward (one
// CTA per row, each phase re-reading the row from global memory, where the
// row stays cached between phases), column sums (repeated passes folding runs
// of 32 rows: the level-by-level tree).

// Tree reduction over i in [0, n) of f(i) (an index functor), as generic_reduce.
template <Op OP, class F>
__device__ float generic_reduce_idx(int64_t n, F f, float *buf, float *buf2, float *bcast) {
    const int runs = int((n + RUN - 1) / RUN);
    for (int j = threadIdx.x; j < runs; j += blockDim.x) {
        const int64_t s = int64_t(j) * RUN, e = imin64(s + RUN, n);
        float acc = f(s);
        for (int64_t i = s + 1; i < e; ++i) acc = combine<OP>(acc, f(i));
        buf[j] = acc;
    }
    return tree_upper<OP>(buf, buf2, runs, bcast);
}

__device__ __forceinline__ float gelu_grad_fixed(float x) {
    const float z = __fmul_rn(x, 0.707106769084930419921875f);
    const float e = erfc_pos(fabsf(z));
    const float phi2 = z >= 0.0f ? __fsub_rn(2.0f, e) : e;
    const float cdf = __fmul_rn(0.5f, phi2);
    const float a = -__fmul_rn(0.5f, __fmul_rn(x, x));
    const float pdf = __fmul_rn(exp_fixed(a), 0.3989422917366028f);   // 1/sqrt(2 pi)
    return __fadd_rn(cdf, __fmul_rn(x, pdf));
}

__global__ void __launch_bounds__(256)
gelu_backward_kernel(int64_t n, const float *__restrict__ x, const float *__restrict__ dy, float *__restrict__ dx,
                     int vec) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const int64_t first = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    int64_t done = 0;
    if (vec) {
        const int64_t n4 = n / 4;
        for (int64_t i = first; i < n4; i += stride) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(x) + i);
            const float4 d = __ldcs(reinterpret_cast<const float4 *>(dy) + i);
            __stcs(reinterpret_cast<float4 *>(dx) + i,
                   make_float4(__fmul_rn(d.x, gelu_grad_fixed(v.x)), __fmul_rn(d.y, gelu_grad_fixed(v.y)),
                               __fmul_rn(d.z, gelu_grad_fixed(v.z)), __fmul_rn(d.w, gelu_grad_fixed(v.w))));
        }
        done = n4 * 4;
    }
    for (int64_t i = done + first; i < n; i += stride) dx[i] = __fmul_rn(dy[i], gelu_grad_fixed(x[i]));
}

// RMSNorm backward: xh = x*inv, gy = dy*gamma, c = tree sum(gy*xh)/n,
// dx = inv*(gy - xh*c) (+ res), p = dy*xh (column sums of p give dgamma).
// res may be dx: each element is read just before it is written.
__global__ void __launch_bounds__(256)
rmsnorm_backward_kernel(int64_t rows, int64_t n, const float *__restrict__ x, int64_t ldx,
                        const float *__restrict__ gamma, float eps, const float *__restrict__ dy, int64_t lddy,
                        const float *res, int64_t ldres, float *dx, int64_t lddx, float *__restrict__ p,
                        int64_t ldp, unsigned *status) {
    extern __shared__ float buf[];
    {
        const int64_t runs = (n + RUN - 1) / RUN;
        if (!REPOPS_DBG_SMEM_OK(uint64_t(runs + (runs + RUN - 1) / RUN) * sizeof(float), status)) return;
    }
    __shared__ float bcast;
    const int runs = int((n + RUN - 1) / RUN);
    float *buf2 = buf + runs;
    const float nf = float(n);
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *xr = x + r * ldx, *dr = dy + r * lddy;
        const float ms = __fdiv_rn(
            generic_reduce_idx<Op::Sum>(n, [&](int64_t i) { return __fmul_rn(xr[i], xr[i]); }, buf, buf2, &bcast),
            nf);
        const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
        const float c = __fdiv_rn(generic_reduce_idx<Op::Sum>(n, [&](int64_t i) {
            return __fmul_rn(__fmul_rn(dr[i], gamma[i]), __fmul_rn(xr[i], inv));
        }, buf, buf2, &bcast), nf);
        for (int j = threadIdx.x; j < runs; j += blockDim.x)
            for (int64_t i = int64_t(j) * RUN; i < imin64(int64_t(j + 1) * RUN, n); ++i) {
                const float xh = __fmul_rn(xr[i], inv), gy = __fmul_rn(dr[i], gamma[i]);
                float d = __fmul_rn(inv, __fsub_rn(gy, __fmul_rn(xh, c)));
                if (res) d = __fadd_rn(d, res[r * ldres + i]);
                dx[r * lddx + i] = d;
                p[r * ldp + i] = __fmul_rn(dr[i], xh);
            }
        __syncthreads();
    }
}

// RMSNorm backward on aligned rows of up to 8192 values, the operations of
// rmsnorm_backward_kernel in the same order: each warp stages its runs of
// the x, dy (and res) rows (coalesced 16-byte copies, swizzled) and gamma once
// per CTA; the two tree reductions fold registers and shuffles; dx and dy*xh
// leave through the x and dy stages.  res may be dx (its row is staged
// before dx is written).
template <int T>
__global__ void __launch_bounds__(T, kNormBwdBlocks<T>)
rmsnorm_backward_staged_kernel(int64_t rows, int64_t n, const float *x, int64_t ldx, const float *gamma, float eps,
                               const float *dy, int64_t lddy, const float *res, int64_t ldres, float *dx,
                               int64_t lddx, float *p, int64_t ldp) {
    extern __shared__ float4 stage_mem[];
    __shared__ float gbuf[2][RUN];
    int phase = 0;
    constexpr int Q = T * RUN / 4;                     // float4 slots per stage
    float4 *sx = stage_mem, *sd = sx + Q, *sg = sd + Q, *sr = sg + Q;
    const int runs = int((n + RUN - 1) / RUN);
    const float nf = float(n);
    if (blockIdx.x < rows) stage_in<T, 1>(sg, gamma, n);   // waited for with the first row
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        stage_in<T, 1>(sx, x + row * ldx, n);
        stage_in<T, 1>(sd, dy + row * lddy, n);
        if (res) stage_in<T, 1>(sr, res + row * ldres, n);
        cp_async_commit();
        cp_async_wait<0>();
        __syncwarp();
        RowRuns<T, 1> a, b;
        read_stage(a, sx, n);
        read_stage(b, sd, n);
        const float ms = __fdiv_rn(a.template reduce<Op::Sum>(Square(), gbuf, phase, runs), nf);
        const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
        const int u = threadIdx.x;
        // gamma and res are read from their stages four values at a time
        // (registers hold the x and dy runs only)
#pragma unroll
        for (int q = 0; q < RUN / 4; ++q) {
            const float4 g4 = sg[stage_slot(u, q)];
            const float g[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int i = 4 * q + t;
                b.v[0][i] = __fmul_rn(__fmul_rn(b.v[0][i], g[t]), __fmul_rn(a.v[0][i], inv));
            }
        }
        const float c = __fdiv_rn(b.template reduce<Op::Sum>(Ident(), gbuf, phase, runs), nf);
        read_stage(b, sd, n);                          // dy again
#pragma unroll
        for (int q = 0; q < RUN / 4; ++q) {
            const float4 g4 = sg[stage_slot(u, q)];
            const float g[4] = {g4.x, g4.y, g4.z, g4.w};
            float r[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (res) {
                const float4 r4 = sr[stage_slot(u, q)];
                r[0] = r4.x; r[1] = r4.y; r[2] = r4.z; r[3] = r4.w;
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int i = 4 * q + t;
                const float xh = __fmul_rn(a.v[0][i], inv), gy = __fmul_rn(b.v[0][i], g[t]);
                float d = __fmul_rn(inv, __fsub_rn(gy, __fmul_rn(xh, c)));
                if (res) d = __fadd_rn(d, r[t]);
                a.v[0][i] = d;
                b.v[0][i] = __fmul_rn(b.v[0][i], xh);
            }
        }
        __syncwarp();                                  // every lane has read its stages before they are rewritten
        write_stage(a, sx);
        write_stage(b, sd);
        __syncwarp();
        stage_out<T, 1>(sx, dx + row * lddx, n);
        stage_out<T, 1>(sd, p + row * ldp, n);
        __syncwarp();
    }
    cp_async_wait<0>();
}

// Values of row r a causal softmax (first, period) saw: all n when first < 0.
__device__ __forceinline__ int64_t causal_prefix(int64_t r, int64_t n, int64_t first, int64_t period) {
    return first < 0 ? n : imin64(n, first + r % period + 1);
}

// Softmax backward over each row's prefix of L values (L = n unless causal):
// s = tree sum(dp*p) over the prefix, ds = p*(dp - s) there and +0 after; the
// entries past the prefix are never read.  Each thread writes only the
// elements it read in the same pass, so ds may be dp or p.
__global__ void __launch_bounds__(256)
softmax_backward_kernel(int64_t rows, int64_t n, const float *p, int64_t ldp, const float *dp, int64_t lddp,
                        float *ds, int64_t ldds, int64_t first, int64_t period, unsigned *status) {
    extern __shared__ float buf[];
    __shared__ float bcast;
    const int runs = int((n + RUN - 1) / RUN);
    if (!REPOPS_DBG_SMEM_OK(uint64_t(runs + (runs + RUN - 1) / RUN) * sizeof(float), status)) return;
    float *buf2 = buf + runs;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *pr = p + r * ldp, *gr = dp + r * lddp;
        const int64_t L = causal_prefix(r, n, first, period);
        const float sum = generic_reduce_idx<Op::Sum>(L, [&](int64_t i) { return __fmul_rn(gr[i], pr[i]); }, buf,
                                                      buf2, &bcast);
        for (int j = threadIdx.x; j < runs; j += blockDim.x)
            for (int64_t i = int64_t(j) * RUN; i < imin64(int64_t(j + 1) * RUN, n); ++i)
                ds[r * ldds + i] = i < L ? __fmul_rn(pr[i], __fsub_rn(gr[i], sum)) : 0.0f;
        __syncthreads();
    }
}

// Softmax backward on aligned rows of up to 8192 values: each warp stages its
// slices of the p and dp rows (coalesced 16-byte copies, swizzled as in the
// forward), each lane folds its run of dp*p, the group fold is by shuffles,
// and ds leaves through the p stage.  dp is read back from its stage after
// the reduction instead of being held in registers.
template <int T>
__global__ void __launch_bounds__(T, kBwdRowBlocks<T>)
softmax_backward_staged_kernel(int64_t rows, int64_t n, const float *p, int64_t ldp, const float *dp, int64_t lddp,
                               float *ds, int64_t ldds, int64_t first, int64_t period) {
    extern __shared__ float4 stage_mem[];
    __shared__ float gbuf[2][RUN];
    int phase = 0;
    float4 *sp = stage_mem, *sd = stage_mem + T * RUN / 4;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        // only the prefix is copied and reduced; the rest of ds is +0
        const int64_t L = causal_prefix(row, n, first, period);
        stage_in<T, 1>(sp, p + row * ldp, L);
        stage_in<T, 1>(sd, dp + row * lddp, L);
        cp_async_commit();
        cp_async_wait<0>();
        __syncwarp();
        RowRuns<T, 1> a, b;
        read_stage(a, sp, L);
        read_stage(b, sd, L);
#pragma unroll
        for (int i = 0; i < RUN; ++i) b.v[0][i] = __fmul_rn(b.v[0][i], a.v[0][i]);   // dp * p
        const float sum = b.template reduce<Op::Sum>(Ident(), gbuf, phase, int((L + RUN - 1) / RUN));
        read_stage(b, sd, L);                                                          // dp again
        const int64_t s0 = int64_t(threadIdx.x) * RUN;
        a.len[0] = s0 < n ? int(imin64(RUN, n - s0)) : 0;
#pragma unroll
        for (int i = 0; i < RUN; ++i)
            a.v[0][i] = s0 + i < L ? __fmul_rn(a.v[0][i], __fsub_rn(b.v[0][i], sum)) : 0.0f;
        __syncwarp();                      // every lane has read both stages before the p stage is rewritten
        write_stage(a, sp);
        __syncwarp();
        stage_out<T, 1>(sp, ds + row * ldds, n);
        __syncwarp();
    }
}

// One tree level of a column sum: out[q][j] = fold of rows [32q, 32q + 32) of
// column j (left to right from the first).  Threads run along columns
// (coalesced), the grid's y dimension along q.
__global__ void __launch_bounds__(256)
colsum_pass_kernel(int64_t rows, int64_t cols, const float *__restrict__ x, int64_t ldx, float *__restrict__ out,
                   int64_t ldo) {
    const int64_t groups = (rows + RUN - 1) / RUN;
    for (int64_t q = blockIdx.y; q < groups; q += gridDim.y) {
        const int64_t r0 = q * RUN, r1 = imin64(r0 + RUN, rows);
        for (int64_t j = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; j < cols;
             j += int64_t(gridDim.x) * blockDim.x) {
            float acc = x[r0 * ldx + j];
            for (int64_t i = r0 + 1; i < r1; ++i) acc = __fadd_rn(acc, x[i * ldx + j]);
            out[q * ldo + j] = acc;
        }
    }
}

// ------------------------------------------------------------ host ----

int check_rows(int64_t rows, int64_t cols, const float *x, int64_t ldx, const float *y, int64_t ldy) {
    if (rows < 0 || cols < 0) return REPOPS_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return REPOPS_OK;
    if (!x || !y || ldx < cols || ldy < cols) return REPOPS_ERR_INVALID_ARG;
    if ((rows - 1) > (INT64_MAX / 4 - cols) / std::max<int64_t>(ldx, ldy)) return REPOPS_ERR_INVALID_ARG;
    if ((cols + RUN - 1) / RUN > MAX_GENERIC_RUNS) return REPOPS_ERR_UNSUPPORTED;
    const uint64_t xb = uint64_t((rows - 1) * ldx + cols) * 4u, yb = uint64_t((rows - 1) * ldy + cols) * 4u;
    // in place (the same rows) is allowed; any other overlap is not
    if (x == y && ldx == ldy) return REPOPS_OK;
    if (ranges_overlap(x, xb, y, yb)) return REPOPS_ERR_ALIAS;
    return REPOPS_OK;
}

bool rows_vec_ok(const float *x, int64_t ldx, const float *y, int64_t ldy) {
    return reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
           ldx % 4 == 0 && ldy % 4 == 0;
}

int grid_for_rows(int64_t rows) {
    DeviceInfo di;
    const int sms = current_device_info(&di) == REPOPS_OK ? di.sms : 152;
    return int(std::min<int64_t>(rows, int64_t(sms) * 32));
}

// Launches `kern` with as many CTAs as fit on the device at once (at most one
// per row); each CTA then strides over the rows.
template <class Kern, class... Args>
int launch_persistent(Kern kern, int threads, size_t smem, int64_t rows, cudaStream_t s, Args... args) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_cuda_error(e);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return set_cuda_error(e);
    DeviceInfo di;
    const int sms = current_device_info(&di) == REPOPS_OK ? di.sms : 152;
    const int grid = int(std::min<int64_t>(rows, int64_t(std::max(per_sm, 1)) * sms));
    kern<<<grid, threads, smem, s>>>(args...);
    return check_launch();
}

// kind 0 = softmax, 1 = LayerNorm, 2 = RMSNorm
template <int T, int R>
int launch_fast(int kind, int64_t rows, int64_t n, const float *x, int64_t ldx, const float *gamma,
                const float *beta, float eps, float *y, int64_t ldy, int64_t first, int64_t period,
                cudaStream_t s) {
    const int pvec = reinterpret_cast<uintptr_t>(gamma) % 16 == 0 && reinterpret_cast<uintptr_t>(beta) % 16 == 0;
    const size_t smem = kStageBytes<T, R>;
    if (kind == 0 && first >= 0)
        return launch_persistent(softmax_causal_rows_kernel<T, R>, T, smem, rows, s, rows, n, x, ldx, y, ldy,
                                 first, period);
    if (kind == 0)
        return launch_persistent(softmax_rows_kernel<T, R>, T, smem, rows, s, rows, n, x, ldx, y, ldy);
    if (kind == 1) {
        const size_t p = pvec ? kParamBytes<T, R, 2> : 0;
        return launch_persistent(layernorm_rows_kernel<T, R>, T, smem + p, rows, s, rows, n, x, ldx, gamma, beta,
                                 eps, y, ldy, pvec, int(p != 0));
    }
    const size_t p = pvec ? kParamBytes<T, R, 1> : 0;
    return launch_persistent(rmsnorm_rows_kernel<T, R>, T, smem + p, rows, s, rows, n, x, ldx, gamma, eps, y, ldy,
                             pvec, int(p != 0));
}

int run_rows(int kind, int64_t rows, int64_t n, const float *x, int64_t ldx, const float *gamma, const float *beta,
             float eps, float *y, int64_t ldy, cudaStream_t s, int64_t first = -1, int64_t period = 1) {
    const int64_t runs = (n + RUN - 1) / RUN;
    // threads per row: enough for one run each up to 256, then up to 4 runs
    // per thread; rows that are not 16-byte aligned, and longer rows, take
    // the long-row kernel (same bits)
    if (rows_vec_ok(x, ldx, y, ldy)) {
        if (runs <= 32) return launch_fast<32, 1>(kind, rows, n, x, ldx, gamma, beta, eps, y, ldy, first, period, s);
        if (runs <= 64) return launch_fast<64, 1>(kind, rows, n, x, ldx, gamma, beta, eps, y, ldy, first, period, s);
        if (runs <= 128) return launch_fast<128, 1>(kind, rows, n, x, ldx, gamma, beta, eps, y, ldy, first, period, s);
        if (runs <= 256) return launch_fast<256, 1>(kind, rows, n, x, ldx, gamma, beta, eps, y, ldy, first, period, s);
        if (runs <= 512) return launch_fast<256, 2>(kind, rows, n, x, ldx, gamma, beta, eps, y, ldy, first, period, s);
        if (runs <= MAX_FAST_RUNS)
            return launch_fast<256, 4>(kind, rows, n, x, ldx, gamma, beta, eps, y, ldy, first, period, s);
    }
    // its shared buffer holds the row's run results and their group results:
    // sized from the row's own run count, whatever the path choice
    const size_t smem = size_t(runs + (runs + RUN - 1) / RUN) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(rows_generic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_cuda_error(e);
    unsigned *status = nullptr;
    int rc = status_word_address(&status);
    if (rc != REPOPS_OK) return rc;
    rows_generic_kernel<<<grid_for_rows(rows), 256, smem, s>>>(kind, rows, n, x, ldx, gamma, beta, eps, y, ldy,
                                                               first, period, status);
    return check_launch();
}

}  // namespace
}  // namespace repops

using namespace repops;

extern "C" int repops_softmax_rows_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y,
                                       int64_t ldy, cudaStream_t stream) {
    int rc = check_rows(rows, cols, x, ldx, y, ldy);
    if (rc != REPOPS_OK || rows == 0 || cols == 0) return rc;
    return run_rows(0, rows, cols, x, ldx, nullptr, nullptr, 0.0f, y, ldy, stream);
}

extern "C" int repops_softmax_rows_causal_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y,
                                              int64_t ldy, int64_t first, int64_t period, cudaStream_t stream) {
    if (first < 0 || period < 1) return REPOPS_ERR_INVALID_ARG;
    int rc = check_rows(rows, cols, x, ldx, y, ldy);
    if (rc != REPOPS_OK || rows == 0 || cols == 0) return rc;
    // from first >= cols on, every row sees all its columns
    if (first < cols && cols <= WARP_CAUSAL_MAX_COLS && rows_vec_ok(x, ldx, y, ldy)) {
        const int row_floats = int((cols + RUN - 1) / RUN * RUN);
        const size_t smem = size_t(WARP_CAUSAL_WARPS) * row_floats * sizeof(float);
        unsigned *status = nullptr;
        if ((rc = status_word_address(&status)) != REPOPS_OK) return rc;
        return launch_persistent(softmax_causal_warp_kernel, 32 * WARP_CAUSAL_WARPS, smem,
                                 (rows + WARP_CAUSAL_WARPS - 1) / WARP_CAUSAL_WARPS, stream, rows, int(cols), x, ldx,
                                 y, ldy, first, period, row_floats, status);
    }
    return run_rows(0, rows, cols, x, ldx, nullptr, nullptr, 0.0f, y, ldy, stream, first < cols ? first : -1,
                    period);
}

extern "C" int repops_layernorm_rows_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                                         const float *gamma, const float *beta, float eps, float *y, int64_t ldy,
                                         cudaStream_t stream) {
    int rc = check_rows(rows, cols, x, ldx, y, ldy);
    if (rc != REPOPS_OK || rows == 0 || cols == 0) return rc;
    if (!gamma || !beta) return REPOPS_ERR_INVALID_ARG;
    const uint64_t yb = uint64_t((rows - 1) * ldy + cols) * 4u;
    if (ranges_overlap(gamma, uint64_t(cols) * 4u, y, yb) || ranges_overlap(beta, uint64_t(cols) * 4u, y, yb))
        return REPOPS_ERR_ALIAS;
    return run_rows(1, rows, cols, x, ldx, gamma, beta, eps, y, ldy, stream);
}

extern "C" int repops_rmsnorm_rows_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                                       const float *gamma, float eps, float *y, int64_t ldy, cudaStream_t stream) {
    int rc = check_rows(rows, cols, x, ldx, y, ldy);
    if (rc != REPOPS_OK || rows == 0 || cols == 0) return rc;
    if (!gamma) return REPOPS_ERR_INVALID_ARG;
    const uint64_t yb = uint64_t((rows - 1) * ldy + cols) * 4u;
    if (ranges_overlap(gamma, uint64_t(cols) * 4u, y, yb)) return REPOPS_ERR_ALIAS;
    return run_rows(2, rows, cols, x, ldx, gamma, nullptr, eps, y, ldy, stream);
}

extern "C" int repops_gelu_f32(int64_t n, const float *x, float *y, cudaStream_t stream) {
    if (n < 0) return REPOPS_ERR_INVALID_ARG;
    if (n == 0) return REPOPS_OK;
    if (!x || !y || n > INT64_MAX / 4) return REPOPS_ERR_INVALID_ARG;
    if (x != y && ranges_overlap(x, uint64_t(n) * 4u, y, uint64_t(n) * 4u)) return REPOPS_ERR_ALIAS;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != REPOPS_OK) return rc;
    const int vec = reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0;
    const int64_t per = vec ? (n + 3) / 4 : n;
    const int grid = int(std::min<int64_t>((per + 255) / 256, int64_t(di.sms) * 8));
    gelu_kernel<<<std::max(grid, 1), 256, 0, stream>>>(n, x, y, vec);
    return check_launch();
}


extern "C" int repops_gelu_backward_f32(int64_t n, const float *x, const float *dy, float *dx, cudaStream_t stream) {
    if (n < 0) return REPOPS_ERR_INVALID_ARG;
    if (n == 0) return REPOPS_OK;
    if (!x || !dy || !dx || n > INT64_MAX / 4) return REPOPS_ERR_INVALID_ARG;
    const uint64_t b = uint64_t(n) * 4u;
    if ((dx != x && ranges_overlap(x, b, dx, b)) || (dx != dy && ranges_overlap(dy, b, dx, b)))
        return REPOPS_ERR_ALIAS;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != REPOPS_OK) return rc;
    const int vec = reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(dy) % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(dx) % 16 == 0;
    const int64_t per = vec ? (n + 3) / 4 : n;
    const int grid = int(std::min<int64_t>((per + 255) / 256, int64_t(di.sms) * 8));
    gelu_backward_kernel<<<std::max(grid, 1), 256, 0, stream>>>(n, x, dy, dx, vec);
    return check_launch();
}

namespace {
// Span check for a rows x cols operand with pitch ld; false on overflow.
bool rows_span(int64_t rows, int64_t cols, int64_t ld, uint64_t *bytes) {
    if (rows == 0 || cols == 0) { *bytes = 0; return true; }
    if (ld < cols || rows - 1 > (INT64_MAX / 4 - cols) / ld) return false;
    *bytes = uint64_t((rows - 1) * ld + cols) * 4u;
    return true;
}
}  // namespace

extern "C" int repops_rmsnorm_backward_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx,
                                           const float *gamma, float eps, const float *dy, int64_t lddy,
                                           const float *res, int64_t ldres, float *dx, int64_t lddx, float *dyxh,
                                           int64_t ldp, cudaStream_t stream) {
    if (rows < 0 || cols < 0) return REPOPS_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return REPOPS_OK;
    if (!x || !gamma || !dy || !dx || !dyxh) return REPOPS_ERR_INVALID_ARG;
    if ((cols + RUN - 1) / RUN > MAX_GENERIC_RUNS) return REPOPS_ERR_UNSUPPORTED;
    uint64_t xb, yb, dxb, pb;
    if (!rows_span(rows, cols, ldx, &xb) || !rows_span(rows, cols, lddy, &yb) || !rows_span(rows, cols, lddx, &dxb) ||
        !rows_span(rows, cols, ldp, &pb))
        return REPOPS_ERR_INVALID_ARG;
    const uint64_t gb = uint64_t(cols) * 4u;
    // outputs are written while every input row is still being re-read: no overlap at all
    for (const void *o : {static_cast<const void *>(dx), static_cast<const void *>(dyxh)})
        for (auto in : {std::make_pair(static_cast<const void *>(x), xb), std::make_pair(static_cast<const void *>(dy), yb),
                        std::make_pair(static_cast<const void *>(gamma), gb)})
            if (ranges_overlap(o, o == dx ? dxb : pb, in.first, in.second)) return REPOPS_ERR_ALIAS;
    if (ranges_overlap(dx, dxb, dyxh, pb)) return REPOPS_ERR_ALIAS;
    if (res) {
        uint64_t rb;
        if (!rows_span(rows, cols, ldres, &rb)) return REPOPS_ERR_INVALID_ARG;
        const bool in_place = res == dx && ldres == lddx;
        if ((!in_place && ranges_overlap(res, rb, dx, dxb)) || ranges_overlap(res, rb, dyxh, pb))
            return REPOPS_ERR_ALIAS;
    }
    const int64_t runs = (cols + RUN - 1) / RUN;
    const bool staged = runs <= 256 && rows_vec_ok(x, ldx, dx, lddx) && rows_vec_ok(dy, lddy, dyxh, ldp) &&
                        reinterpret_cast<uintptr_t>(gamma) % 16 == 0 && (!res || rows_vec_ok(res, ldres, dx, lddx));
    if (staged) {
        auto go = [&](auto kern, int T) {
            return launch_persistent(kern, T, size_t(4) * T * RUN * sizeof(float), rows, stream, rows, cols, x, ldx,
                                     gamma, eps, dy, lddy, res, ldres, dx, lddx, dyxh, ldp);
        };
        if (runs <= 32) return go(rmsnorm_backward_staged_kernel<32>, 32);
        if (runs <= 64) return go(rmsnorm_backward_staged_kernel<64>, 64);
        if (runs <= 128) return go(rmsnorm_backward_staged_kernel<128>, 128);
        return go(rmsnorm_backward_staged_kernel<256>, 256);
    }
    const size_t smem = size_t(runs + (runs + RUN - 1) / RUN) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(rmsnorm_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_cuda_error(e);
    unsigned *status = nullptr;
    if (status_word_address(&status) != REPOPS_OK) status = nullptr;
    rmsnorm_backward_kernel<<<grid_for_rows(rows), 256, smem, stream>>>(rows, cols, x, ldx, gamma, eps, dy, lddy, res,
                                                                         ldres, dx, lddx, dyxh, ldp, status);
    return check_launch();
}

namespace {
int softmax_backward(int64_t rows, int64_t cols, const float *p, int64_t ldp, const float *dp, int64_t lddp,
                     float *ds, int64_t ldds, int64_t first, int64_t period, cudaStream_t stream) {
    if (rows < 0 || cols < 0) return REPOPS_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return REPOPS_OK;
    if (!p || !dp || !ds) return REPOPS_ERR_INVALID_ARG;
    if ((cols + RUN - 1) / RUN > MAX_GENERIC_RUNS) return REPOPS_ERR_UNSUPPORTED;
    uint64_t pb, gb, sb;
    if (!rows_span(rows, cols, ldp, &pb) || !rows_span(rows, cols, lddp, &gb) || !rows_span(rows, cols, ldds, &sb))
        return REPOPS_ERR_INVALID_ARG;
    // in place over p or dp (same pitch) is allowed: each element is written after its last read
    const bool on_p = ds == p && ldds == ldp, on_dp = ds == dp && ldds == lddp;
    if ((!on_p && ranges_overlap(ds, sb, p, pb)) || (!on_dp && ranges_overlap(ds, sb, dp, gb))) return REPOPS_ERR_ALIAS;
    const int64_t runs = (cols + RUN - 1) / RUN;
    const bool staged = runs <= 256 && rows_vec_ok(p, ldp, ds, ldds) && rows_vec_ok(dp, lddp, ds, ldds);
    if (staged) {
        auto go = [&](auto kern, int T) {
            return launch_persistent(kern, T, size_t(2) * T * RUN * sizeof(float), rows, stream, rows, cols, p,
                                     ldp, dp, lddp, ds, ldds, first, period);
        };
        if (runs <= 32) return go(softmax_backward_staged_kernel<32>, 32);
        if (runs <= 64) return go(softmax_backward_staged_kernel<64>, 64);
        if (runs <= 128) return go(softmax_backward_staged_kernel<128>, 128);
        return go(softmax_backward_staged_kernel<256>, 256);
    }
    const size_t smem = size_t(runs + (runs + RUN - 1) / RUN) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(softmax_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_cuda_error(e);
    unsigned *status = nullptr;
    if (status_word_address(&status) != REPOPS_OK) status = nullptr;
    softmax_backward_kernel<<<grid_for_rows(rows), 256, smem, stream>>>(rows, cols, p, ldp, dp, lddp, ds, ldds,
                                                                        first, period, status);
    return check_launch();
}
}  // namespace

extern "C" int repops_softmax_backward_f32(int64_t rows, int64_t cols, const float *p, int64_t ldp, const float *dp,
                                           int64_t lddp, float *ds, int64_t ldds, cudaStream_t stream) {
    return softmax_backward(rows, cols, p, ldp, dp, lddp, ds, ldds, -1, 1, stream);
}

extern "C" int repops_softmax_backward_causal_f32(int64_t rows, int64_t cols, const float *p, int64_t ldp,
                                                  const float *dp, int64_t lddp, float *ds, int64_t ldds,
                                                  int64_t first, int64_t period, cudaStream_t stream) {
    if (first < 0 || period < 1) return REPOPS_ERR_INVALID_ARG;
    // from first >= cols - 1 on, every row's prefix is the whole row
    return softmax_backward(rows, cols, p, ldp, dp, lddp, ds, ldds, first < cols - 1 ? first : -1, period, stream);
}

extern "C" int repops_colsum_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y,
                                 cudaStream_t stream) {
    if (rows < 0 || cols < 0) return REPOPS_ERR_INVALID_ARG;
    if (cols == 0) return REPOPS_OK;
    if (!y) return REPOPS_ERR_INVALID_ARG;
    if (rows == 0) {   // an empty column sums to +0
        cudaError_t e = cudaMemsetAsync(y, 0, size_t(cols) * 4u, stream);
        return e == cudaSuccess ? REPOPS_OK : set_cuda_error(e);
    }
    uint64_t xb;
    if (!x || !rows_span(rows, cols, ldx, &xb)) return REPOPS_ERR_INVALID_ARG;
    if (ranges_overlap(x, xb, y, uint64_t(cols) * 4u)) return REPOPS_ERR_ALIAS;
    // scratch for the levels between the input and y: ceil(rows/32) rows, then ceil(rows/1024), ...
    int64_t need = 0;
    for (int64_t r = (rows + RUN - 1) / RUN; r > 1; r = (r + RUN - 1) / RUN) need += r;
    float *scratch = nullptr;
    if (need > 0) {
        if (scratch_malloc(reinterpret_cast<void **>(&scratch), size_t(need) * size_t(cols) * 4u, stream) != cudaSuccess) {
            cudaGetLastError();
            return REPOPS_ERR_ALLOC;
        }
    }
    int rc = REPOPS_OK;
    const float *in = x;
    int64_t in_rows = rows, in_ld = ldx;
    float *level = scratch;
    while (rc == REPOPS_OK) {
        const int64_t out_rows = (in_rows + RUN - 1) / RUN;
        float *out = out_rows == 1 ? y : level;   // every level is packed: pitch cols
        const int gx = int(std::min<int64_t>((cols + 255) / 256, 64));
        const int gy = int(std::min<int64_t>(out_rows, 65535));
        colsum_pass_kernel<<<dim3(gx, gy), 256, 0, stream>>>(in_rows, cols, in, in_ld, out, cols);
        rc = check_launch();
        if (out_rows == 1) break;
        in = out;
        in_rows = out_rows;
        in_ld = cols;
        level += out_rows * cols;
    }
    if (scratch) {
        cudaError_t e = cudaFreeAsync(scratch, stream);
        if (rc == REPOPS_OK && e != cudaSuccess) rc = set_cuda_error(e);
    }
    return rc;
}
