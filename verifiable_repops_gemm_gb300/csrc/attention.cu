// attention.cu -- fused causal attention for one head dimension of 64: the
// scores, the causal softmax and the banded product with V of a block of query
// rows in one CTA, the scores and probabilities kept in shared memory.
//
// What is computed is the library's causal attention, step by step the same
// operations as its unfused form ("Verde与RepOps" §3.2: order-critical
// reductions keep one fixed order; §4.3: the Llama-1B training measurement):
//   s[i][j] = fl(scale * acc), acc = the k-chain over d = 0 .. 63 of
//             fl(q_i[d] * k_j[d]) from +0 (repops_gemm_f32_batched with alpha;
//             scale == 1 skips the multiply, which is exact);
//   p[i][.] = the causal softmax of row i over its prefix j <= i
//             (repops_softmax_rows_causal_f32: the 32-ary max and sum trees,
//             the library's exp, one correctly rounded reciprocal), +0 after;
//   o[i][c] = the chain over j = 0 .. i of fl(p[i][j] * v_j[c]) from +0 (the
//             banded product of repops_gemm_f32_batched with k_hi = 0).
// Products past a row's prefix are not added at all (a select, not a multiply
// by +0), so the result is that definition for any V, finite or not.
//
// One CTA = one query head of one sequence x 16 consecutive query rows; rows
// [i0, i0 + 16) need keys [0, L), L = min(S, i0 + 16).  Keys and values are
// streamed through a double-buffered shared-memory ring in chunks of 128 rows
// (cp.async, 16 bytes per copy).  Phase 1: every score of the block (the
// d-chains run in registers, 2 rows x 4 keys a thread, products paired by
// packed adds as in the GEMM); phase 2: one warp per row folds the trees by
// runs and shuffles and exponentiates in place; phase 3: the p-v chains, 2 rows
// x 2 columns a thread.  Scores live in a 16 x 2048 array whose 32-value runs
// are XOR-swizzled in 16-byte groups, so that a lane per run reads without
// bank conflicts and float4 groups of consecutive keys stay contiguous.
#include <algorithm>
#include <cstdint>

#include "fixed_math.cuh"
#include "internal.cuh"

namespace repops {
namespace {

constexpr int ABM = 16;          // query rows per CTA
constexpr int ACH = 128;         // keys per chunk
constexpr int ADH = 64;          // head dimension
constexpr int ATHREADS = 256;    // 8 warps
constexpr int AMAXS = 2048;      // longest sequence (scores of a row in shared memory)
constexpr int KST = ADH + 4;     // padded row stride of a key/value chunk (floats)
constexpr int QST = ADH + 4;     // padded row stride of the query block
constexpr int PST = AMAXS + 4;   // padded row stride of the scores: rows 4 banks apart

constexpr size_t kPsFloats = size_t(ABM) * PST;
constexpr size_t kQsFloats = size_t(ABM) * QST;
constexpr size_t kKvFloats = size_t(ACH) * KST;
constexpr size_t kAttnSmem = (kPsFloats + kQsFloats + 2 * kKvFloats) * 4;

// Position of key j of a row inside its score row: 16-byte groups of a 32-value
// run permuted by the run index (a group keeps its 4 consecutive keys).
__device__ __forceinline__ int ps_pos(int j) { return (j & ~31) | ((j & 31) ^ (((j >> 5) & 7) << 2)); }

struct AttnArgs {
    const float *q, *k, *v;
    int64_t ldq, ldk, ldv;
    float *out;
    int64_t ldo;
    float *probs;        // (seqs * heads, S, S) or null
    int seqs, S, heads, group;
    float scale;
    int row_blocks;
};

// Copies rows [r0, r0 + n) (n <= rows) of 64 floats at `src` (pitch ld) into
// shared memory at pitch `st`; rows at or past `valid` are filled with zeros.
template <int ROWS>
__device__ __forceinline__ void load_rows64(float *dst, int st, const float *__restrict__ src, int64_t ld, int r0,
                                            int valid) {
    constexpr int COPIES = ROWS * (ADH / 4);
#pragma unroll
    for (int c = threadIdx.x; c < COPIES; c += ATHREADS) {
        const int r = c >> 4, part = c & 15;
        const bool ok = r0 + r < valid;
        const float *s = ok ? src + int64_t(r0 + r) * ld + part * 4 : src;
        cp_async_16(dst + r * st + part * 4, s, ok ? 16u : 0u);
    }
}

// The tree fold of one row's run results across the warp: lane l holds run
// (32g + l)'s result for group g = 0, 1; runs >= nruns are absent.  Every lane
// returns the root (groups folded left to right by shuffles, then the group
// results left to right).
template <bool MAX>
__device__ __forceinline__ float warp_tree_top(float r0, float r1, int nruns) {
    float root = 0.0f;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int have = nruns - 32 * g;
        if (have <= 0) break;               // warp-uniform
        const float mine = g == 0 ? r0 : r1;
        float acc = __shfl_sync(0xffffffffu, mine, 0);
#pragma unroll
        for (int i = 1; i < 32; ++i) {
            const float o = __shfl_sync(0xffffffffu, mine, i);
            if (i < have) acc = MAX ? (o > acc ? o : acc) : __fadd_rn(acc, o);
        }
        if (g == 0) root = acc;
        else root = MAX ? (acc > root ? acc : root) : __fadd_rn(root, acc);
    }
    return root;
}

__global__ void __launch_bounds__(ATHREADS, 1) attention_causal_kernel(const AttnArgs a) {
    extern __shared__ float4 attn_smem4[];
    float *Ps = reinterpret_cast<float *>(attn_smem4);
    float *Qs = Ps + kPsFloats;
    float *KV0 = Qs + kQsFloats;
    float *KV1 = KV0 + kKvFloats;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lm = lane >> 3, ln = lane & 7;
    const int sh_count = a.seqs * a.heads;
    const int rb = a.row_blocks - 1 - int(blockIdx.x / sh_count);   // longest blocks first
    const int sh = int(blockIdx.x % sh_count);
    const int seq = sh / a.heads, h = sh % a.heads, g = h / a.group;
    const int S = a.S;
    const int i0 = rb * ABM;
    const int L = min(S, i0 + ABM);                 // keys any row of the block needs
    const int nch = (L + ACH - 1) / ACH;
    const int64_t row0 = int64_t(seq) * S;          // the sequence's first row
    const float *qb = a.q + row0 * a.ldq + int64_t(h) * ADH;
    const float *kb = a.k + row0 * a.ldk + int64_t(g) * ADH;
    const float *vb = a.v + row0 * a.ldv + int64_t(g) * ADH;

    // ---------------------------------------------------------- scores ----
    const int warp_m = warp & 1, warp_n = warp >> 1;
    const int qr0 = warp_m * 8 + lm;                // rows qr0 and qr0 + 4
    const int kc0 = warp_n * 32 + ln;               // keys kc0 + 8c of a chunk

    load_rows64<ABM>(Qs, QST, qb, a.ldq, i0, S);
    load_rows64<ACH>(KV0, KST, kb, a.ldk, 0, L);
    cp_async_commit();
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
        float *cur = (c & 1) ? KV1 : KV0;
        if (c + 1 < nch) load_rows64<ACH>((c & 1) ? KV0 : KV1, KST, kb, a.ldk, (c + 1) * ACH, L);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        u64 acc[2][2];
#pragma unroll
        for (int r = 0; r < 2; ++r) acc[r][0] = acc[r][1] = 0ull;   // +0
#pragma unroll
        for (int d4 = 0; d4 < ADH / 4; ++d4) {
            float qv[2][4], kv[4][4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float4 t = *reinterpret_cast<const float4 *>(Qs + (qr0 + 4 * r) * QST + 4 * d4);
                qv[r][0] = t.x; qv[r][1] = t.y; qv[r][2] = t.z; qv[r][3] = t.w;
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const float4 t = *reinterpret_cast<const float4 *>(cur + (kc0 + 8 * cc) * KST + 4 * d4);
                kv[cc][0] = t.x; kv[cc][1] = t.y; kv[cc][2] = t.z; kv[cc][3] = t.w;
            }
#pragma unroll
            for (int dd = 0; dd < 4; ++dd)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    acc[r][0] = fold2(acc[r][0], qv[r][dd], kv[0][dd], qv[r][dd], kv[1][dd]);
                    acc[r][1] = fold2(acc[r][1], qv[r][dd], kv[2][dd], qv[r][dd], kv[3][dd]);
                }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float s[4];
            unpack2(acc[r][0], s[0], s[1]);
            unpack2(acc[r][1], s[2], s[3]);
            float *prow = Ps + (qr0 + 4 * r) * PST;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int j = c * ACH + kc0 + 8 * cc;
                if (j < L) prow[ps_pos(j)] = a.scale == 1.0f ? s[cc] : __fmul_rn(a.scale, s[cc]);
            }
        }
        __syncthreads();   // `cur` is refilled by the next iteration's copies
    }

    // the first value chunk streams in while the softmax runs
    load_rows64<ACH>(KV0, KST, vb, a.ldv, 0, L);
    cp_async_commit();

    // --------------------------------------------------------- softmax ----
    // warp w: rows w and w + 8; lane l: runs l and l + 32 of a row
#pragma unroll 1
    for (int rr = 0; rr < 2; ++rr) {
        const int r = warp + 8 * rr, i = i0 + r;
        if (i >= S) continue;                       // warp-uniform
        float *prow = Ps + r * PST;
        const int Li = i + 1, nruns = (Li + 31) >> 5;
        float rm[2] = {0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int u = lane + 32 * k;
            if (u >= nruns) continue;
            const int len = min(32, Li - 32 * u);
            const float *run = prow + 32 * u;
            float m = 0.0f;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 t = *reinterpret_cast<const float4 *>(run + 4 * (q4 ^ (u & 7)));
                const float v4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int idx = 4 * q4 + e;
                    if (idx == 0) m = v4[0];
                    else if (idx < len && v4[e] > m) m = v4[e];
                }
            }
            rm[k] = m;
        }
        const float mx = warp_tree_top<true>(rm[0], rm[1], nruns);
        __syncwarp();                               // every run read before it is overwritten
        // exponentials of the prefix, spread over every lane (4 consecutive
        // keys a lane at a time), written in place
        for (int j4 = 4 * lane; j4 < Li; j4 += 128) {
            float4 *p4 = reinterpret_cast<float4 *>(prow + ps_pos(j4));
            float4 t = *p4;
            float d0, d1, d2, d3;
            unpack2(add2_rn(pack2(t.x, t.y), pack2(-mx, -mx)), d0, d1);
            unpack2(add2_rn(pack2(t.z, t.w), pack2(-mx, -mx)), d2, d3);
            const float2 e01 = exp_fixed2(d0, d1), e23 = exp_fixed2(d2, d3);
            *p4 = make_float4(e01.x, e01.y, e23.x, e23.y);
        }
        __syncwarp();
        // the sum tree: each lane folds its runs left to right
        float rs[2] = {0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int u = lane + 32 * k;
            if (u >= nruns) continue;
            const int len = min(32, Li - 32 * u);
            const float *run = prow + 32 * u;
            float sum = 0.0f;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 t = *reinterpret_cast<const float4 *>(run + 4 * (q4 ^ (u & 7)));
                const float e4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int idx = 4 * q4 + e;
                    if (idx == 0) sum = e4[0];
                    else if (idx < len) sum = __fadd_rn(sum, e4[e]);
                }
            }
            rs[k] = sum;
        }
        const float inv = __frcp_rn(warp_tree_top<false>(rs[0], rs[1], nruns));
        __syncwarp();
        // p = e * inv inside the prefix; +0 from the prefix to the end of the
        // block's keys (the product phase selects by row, but a full row is
        // what the probabilities output holds)
        const int lend = nch * ACH;
        for (int j4 = 4 * lane; j4 < lend; j4 += 128) {
            float4 *p4 = reinterpret_cast<float4 *>(prow + ps_pos(j4));
            float4 t = *p4;
            t.x = j4 + 0 < Li ? __fmul_rn(t.x, inv) : 0.0f;
            t.y = j4 + 1 < Li ? __fmul_rn(t.y, inv) : 0.0f;
            t.z = j4 + 2 < Li ? __fmul_rn(t.z, inv) : 0.0f;
            t.w = j4 + 3 < Li ? __fmul_rn(t.w, inv) : 0.0f;
            *p4 = t;
        }
        if (a.probs) {
            __syncwarp();
            float *dst = a.probs + (int64_t(sh) * S + i) * S;
            for (int j4 = 4 * lane; j4 < S; j4 += 128) {
                float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (j4 < Li) t = *reinterpret_cast<const float4 *>(prow + ps_pos(j4));
                __stcs(reinterpret_cast<float4 *>(dst + j4), t);
            }
        }
    }
    __syncthreads();

    // --------------------------------------------------------- p * v ----
    const int pr0 = warp_m * 8 + lm;                // rows pr0 and pr0 + 4
    const int vc = warp_n * 16 + 2 * ln;            // columns vc and vc + 1
    const int irow[2] = {i0 + pr0, i0 + pr0 + 4};
    u64 o[2] = {0ull, 0ull};
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
        const float *cur = (c & 1) ? KV1 : KV0;
        if (c + 1 < nch) load_rows64<ACH>((c & 1) ? KV0 : KV1, KST, vb, a.ldv, (c + 1) * ACH, L);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int j0 = c * ACH;
        // keys past a row's prefix are skipped only in the chunk that holds
        // the block's diagonal
        const bool diag = j0 + ACH - 1 > i0;
        if (!diag) {
#pragma unroll 1
            for (int u = 0; u < ACH / 32; ++u) {
                // run R of the row: its 16-byte groups are permuted by R & 7
                const int R = (j0 >> 5) + u, key = (R & 7) << 2;
                const float *p0 = Ps + pr0 * PST + 32 * R;
                const float *vrow = cur + 32 * u * KST + vc;
#pragma unroll
                for (int a8 = 0; a8 < 8; ++a8) {
                    const int off = (4 * a8) ^ key;
                    const float4 t0 = *reinterpret_cast<const float4 *>(p0 + off);
                    const float4 t1 = *reinterpret_cast<const float4 *>(p0 + 4 * PST + off);
                    const float pv[2][4] = {{t0.x, t0.y, t0.z, t0.w}, {t1.x, t1.y, t1.z, t1.w}};
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float2 v2 = *reinterpret_cast<const float2 *>(vrow + (4 * a8 + jj) * KST);
#pragma unroll
                        for (int r = 0; r < 2; ++r) o[r] = fold2(o[r], pv[r][jj], v2.x, pv[r][jj], v2.y);
                    }
                }
            }
        } else {
#pragma unroll 1
            for (int j4 = 0; j4 < ACH / 4; ++j4) {
                float pv[2][4];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float4 t =
                        *reinterpret_cast<const float4 *>(Ps + (pr0 + 4 * r) * PST + ps_pos(j0 + 4 * j4));
                    pv[r][0] = t.x; pv[r][1] = t.y; pv[r][2] = t.z; pv[r][3] = t.w;
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = j0 + 4 * j4 + jj;
                    const float2 v2 = *reinterpret_cast<const float2 *>(cur + (4 * j4 + jj) * KST + vc);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        // a term past the row's prefix is not added: +0 leaves
                        // the accumulator (never -0) unchanged
                        const bool in = j <= irow[r];
                        const u64 prod = in ? pack2(__fmul_rn(pv[r][jj], v2.x), __fmul_rn(pv[r][jj], v2.y)) : 0ull;
                        o[r] = add2_rn(o[r], prod);
                    }
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (irow[r] >= S) continue;
        float x0, x1;
        unpack2(o[r], x0, x1);
        float *dst = a.out + (row0 + irow[r]) * a.ldo + int64_t(h) * ADH + vc;
        dst[0] = x0;
        dst[1] = x1;
    }
}

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace
}  // namespace repops

using namespace repops;

extern "C" int repops_attention_causal_f32(int64_t seqs, int64_t S, int64_t heads, int64_t kv_heads, int64_t dh,
                                           const float *q, int64_t ldq, const float *k, int64_t ldk,
                                           const float *v, int64_t ldv, float scale, float *out, int64_t ldo,
                                           float *probs, cudaStream_t stream) {
    if (seqs < 0 || S < 0 || heads < 0 || kv_heads < 0 || dh < 0) return REPOPS_ERR_INVALID_ARG;
    if (seqs == 0 || S == 0 || heads == 0) return REPOPS_OK;
    if (kv_heads == 0 || heads % kv_heads != 0) return REPOPS_ERR_INVALID_ARG;
    if (!q || !k || !v || !out) return REPOPS_ERR_INVALID_ARG;
    // the limits first: they bound every product below
    if (dh != ADH || S > AMAXS) return REPOPS_ERR_UNSUPPORTED;
    if (heads > (int64_t(1) << 31) || seqs > (int64_t(1) << 31) / heads || seqs * S > (int64_t(1) << 40))
        return REPOPS_ERR_UNSUPPORTED;
    if (ldq < heads * dh || ldk < kv_heads * dh || ldv < kv_heads * dh || ldo < heads * dh)
        return REPOPS_ERR_INVALID_ARG;
    // 16-byte copies of every query, key and value row; float4 rows of probs
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || ldq % 4 || ldk % 4 || ldv % 4 || ldo % 2 ||
        reinterpret_cast<uintptr_t>(out) % 8 || (probs && (!aligned16(probs) || S % 4)))
        return REPOPS_ERR_UNSUPPORTED;
    const int64_t rows = seqs * S;
    const uint64_t ob = (uint64_t(rows - 1) * uint64_t(ldo) + uint64_t(heads * dh)) * 4u;
    const uint64_t qbytes = (uint64_t(rows - 1) * uint64_t(ldq) + uint64_t(heads * dh)) * 4u;
    const uint64_t kbytes = (uint64_t(rows - 1) * uint64_t(ldk) + uint64_t(kv_heads * dh)) * 4u;
    const uint64_t vbytes = (uint64_t(rows - 1) * uint64_t(ldv) + uint64_t(kv_heads * dh)) * 4u;
    if (ranges_overlap(out, ob, q, qbytes) || ranges_overlap(out, ob, k, kbytes) ||
        ranges_overlap(out, ob, v, vbytes))
        return REPOPS_ERR_ALIAS;
    if (probs) {
        const uint64_t pb = uint64_t(seqs * heads) * uint64_t(S) * uint64_t(S) * 4u;
        if (ranges_overlap(probs, pb, q, qbytes) || ranges_overlap(probs, pb, k, kbytes) ||
            ranges_overlap(probs, pb, v, vbytes) || ranges_overlap(probs, pb, out, ob))
            return REPOPS_ERR_ALIAS;
    }
    AttnArgs a;
    a.q = q; a.k = k; a.v = v;
    a.ldq = ldq; a.ldk = ldk; a.ldv = ldv;
    a.out = out; a.ldo = ldo;
    a.probs = probs;
    a.seqs = int(seqs); a.S = int(S); a.heads = int(heads); a.group = int(heads / kv_heads);
    a.scale = scale;
    a.row_blocks = int((S + ABM - 1) / ABM);
    const int64_t blocks = int64_t(a.row_blocks) * seqs * heads;
    if (blocks > 0x7fffffffLL) return REPOPS_ERR_UNSUPPORTED;
    cudaError_t e = cudaFuncSetAttribute(attention_causal_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kAttnSmem));
    if (e != cudaSuccess) return set_cuda_error(e);
    attention_causal_kernel<<<unsigned(blocks), ATHREADS, kAttnSmem, stream>>>(a);
    return check_launch();
}
