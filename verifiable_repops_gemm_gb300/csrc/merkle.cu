// merkle.cu -- SHA-256 Merkle commitment over tensor bytes.
//
// "Zoo Per-LLM Chain Soundness" §1 (a block carries the Merkle root of its
// input batch and the model state root), §6 (roots are bytes32), §7 (a
// replaying party checks H(theta) = m); "Verde与RepOps" §2.3.2 (checkpoint
// hashes are Merkle trees over node hashes) and §2.4 (Merkle membership
// proofs).  The pages name no hash function or encoding; the library takes
//   leaf = SHA256(0x00 || leaf bytes), node = SHA256(0x01 || left || right),
// leaves of `leaf` bytes in increasing offset (the last may be short), levels
// reduced pairwise with an unpaired last node promoted unchanged.  SHA-256 is
// FIPS 180-4.
//
// Kernels:
//   merkle_leaf_subtree: one leaf per thread (65 compressions for a 4 KiB
//     leaf), then the CTA folds its LEAF_CTA leaves into the level-log2(LEAF_CTA)
//     node in shared memory.  Node j of level l covers leaves [j*2^l,
//     (j+1)*2^l), so a CTA-aligned block of leaves reduces to exactly that
//     node, promotion included.
//   merkle_reduce: each CTA folds up to 2*RED_CTA consecutive nodes of a level
//     into one; repeated until one node, the root, remains.
// SHA-256 is bound by the integer ALU (about 22 integer instructions per
// message byte), far below HBM bandwidth.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.cuh"

namespace repops {
namespace {

constexpr int LEAF_CTA = 128;   // leaves per CTA in the leaf kernel (power of two)
constexpr int LOG_LEAF_CTA = 7;
constexpr int RED_CTA = 256;    // threads per CTA in the reduce kernel
constexpr int LOG_RED_NODES = 9;   // a reduce CTA folds 2 * RED_CTA = 2^9 nodes
static_assert((1 << LOG_LEAF_CTA) == LEAF_CTA && (1 << LOG_RED_NODES) == 2 * RED_CTA, "fold depths");

// FIPS 180-4 §4.2.2: first 32 bits of the fractional parts of the cube roots
// of the first 64 primes.
__constant__ uint32_t c_K[64] = {
    0x428a2f98u, 0x71374491u, 0xb5c0fbcfu, 0xe9b5dba5u, 0x3956c25bu, 0x59f111f1u, 0x923f82a4u, 0xab1c5ed5u,
    0xd807aa98u, 0x12835b01u, 0x243185beu, 0x550c7dc3u, 0x72be5d74u, 0x80deb1feu, 0x9bdc06a7u, 0xc19bf174u,
    0xe49b69c1u, 0xefbe4786u, 0x0fc19dc6u, 0x240ca1ccu, 0x2de92c6fu, 0x4a7484aau, 0x5cb0a9dcu, 0x76f988dau,
    0x983e5152u, 0xa831c66du, 0xb00327c8u, 0xbf597fc7u, 0xc6e00bf3u, 0xd5a79147u, 0x06ca6351u, 0x14292967u,
    0x27b70a85u, 0x2e1b2138u, 0x4d2c6dfcu, 0x53380d13u, 0x650a7354u, 0x766a0abbu, 0x81c2c92eu, 0x92722c85u,
    0xa2bfe8a1u, 0xa81a664bu, 0xc24b8b70u, 0xc76c51a3u, 0xd192e819u, 0xd6990624u, 0xf40e3585u, 0x106aa070u,
    0x19a4c116u, 0x1e376c08u, 0x2748774cu, 0x34b0bcb5u, 0x391c0cb3u, 0x4ed8aa4au, 0x5b9cca4fu, 0x682e6ff3u,
    0x748f82eeu, 0x78a5636fu, 0x84c87814u, 0x8cc70208u, 0x90befffau, 0xa4506cebu, 0xbef9a3f7u, 0xc67178f2u};

// FIPS 180-4 §5.3.3: first 32 bits of the fractional parts of the square roots
// of the first 8 primes.
__constant__ uint32_t c_H0[8] = {0x6a09e667u, 0xbb67ae85u, 0x3c6ef372u, 0xa54ff53au,
                                 0x510e527fu, 0x9b05688cu, 0x1f83d9abu, 0x5be0cd19u};

__device__ __forceinline__ uint32_t rotr(uint32_t x, int n) { return __funnelshift_r(x, x, n); }

// SHA-256 is bound by the integer ALU pipe, which issues at half rate, while
// the pipe that runs integer multiply-adds idles.  So every 32-bit addition is
// written x * one + y, with `one` a kernel argument the compiler cannot fold
// back into an add: those instructions run on the multiply-add pipe.  Same
// arithmetic mod 2^32, same bits.  (Measured on 4 GiB: 869 -> 1008 GB/s
// together with the 16-round loop body below.  Moving more there is slower:
// the schedule's shifts as high halves of products 1008 -> 1020 GB/s when
// taken back to the ALU, a rotate of a sigma as two products -3%, a
// three-input sum as one ALU add instead of two multiply-adds -1 to -4%, two
// rotates of each Sigma as the two halves of one 64-bit product each (one
// ALU operation fewer per Sigma) -18%.)
struct PipeConst {
    uint32_t one;     // 1
};

__device__ __forceinline__ uint32_t add_u(uint32_t x, uint32_t y, const PipeConst &c) { return x * c.one + y; }

// One round of FIPS 180-4 §6.2.2 with message word w and constant k.
__device__ __forceinline__ void sha256_round(uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d,
                                             uint32_t &e, uint32_t &f, uint32_t &g, uint32_t &h,
                                             uint32_t w, uint32_t k, const PipeConst &pc) {
    // h + K[t] + w does not depend on this round's e: off the critical path
    const uint32_t hkw = add_u(add_u(h, w, pc), k, pc);
    const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    const uint32_t ch = (e & f) ^ (~e & g);
    const uint32_t T1 = add_u(add_u(S1, ch, pc), hkw, pc);
    const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
    const uint32_t T2 = add_u(S0, maj, pc);
    h = g; g = f; f = e; e = add_u(d, T1, pc);
    d = c; c = b; b = a; a = add_u(T1, T2, pc);
}

// FIPS 180-4 §6.2.2 for one 512-bit block held as 16 big-endian words in W
// (W is used as the rolling message schedule and is clobbered).  Rounds run in
// 16-round unrolled bodies: the schedule's slots stay static while the loop
// body (~7 KB) fits the instruction cache; a fully unrolled 64-round body
// stalled on instruction fetch.
__device__ __forceinline__ void sha256_compress(uint32_t (&st)[8], uint32_t (&W)[16], const PipeConst &pc) {
    uint32_t a = st[0], b = st[1], c = st[2], d = st[3];
    uint32_t e = st[4], f = st[5], g = st[6], h = st[7];
#pragma unroll
    for (int j = 0; j < 16; ++j) sha256_round(a, b, c, d, e, f, g, h, W[j], c_K[j], pc);
#pragma unroll 1
    for (int t0 = 16; t0 < 64; t0 += 16) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            // W_t = s1(W_{t-2}) + W_{t-7} + s0(W_{t-15}) + W_{t-16}, in place: slot j holds W_{t-16}
            const uint32_t x = W[(j + 1) & 15], y = W[(j + 14) & 15];
            const uint32_t s0 = rotr(x, 7) ^ rotr(x, 18) ^ (x >> 3);
            const uint32_t s1 = rotr(y, 17) ^ rotr(y, 19) ^ (y >> 10);
            const uint32_t w = add_u(add_u(add_u(s1, W[(j + 9) & 15], pc), s0, pc), W[j], pc);
            W[j] = w;
            sha256_round(a, b, c, d, e, f, g, h, w, c_K[t0 + j], pc);
        }
    }
    st[0] = add_u(st[0], a, pc); st[1] = add_u(st[1], b, pc);
    st[2] = add_u(st[2], c, pc); st[3] = add_u(st[3], d, pc);
    st[4] = add_u(st[4], e, pc); st[5] = add_u(st[5], f, pc);
    st[6] = add_u(st[6], g, pc); st[7] = add_u(st[7], h, pc);
}

__device__ __forceinline__ void sha256_init(uint32_t (&st)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) st[i] = c_H0[i];
}

// Digest of a full, 16-byte aligned leaf of `leaf` bytes (a multiple of 64):
// the message 0x00 || data is shifted one byte against the data, so message
// word t of block b is bytes [64b + 4t - 1, 64b + 4t + 3) of the data, built
// from two little-endian data words with one byte permute.
__device__ __forceinline__ void leaf_digest_fast(const uint8_t *__restrict__ p, uint32_t leaf,
                                                 uint32_t (&st)[8], const PipeConst &pc) {
    sha256_init(st);
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    uint32_t prev = 0;   // byte 3 of "word -1" is the 0x00 prefix
    const uint32_t nblk = leaf / 64;
#pragma unroll 1
    for (uint32_t blk = 0; blk < nblk; ++blk) {
        uint32_t d[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 x = __ldcs(q + 4 * blk + v);
            d[4 * v] = x.x; d[4 * v + 1] = x.y; d[4 * v + 2] = x.z; d[4 * v + 3] = x.w;
        }
        uint32_t W[16];
        W[0] = __byte_perm(prev, d[0], 0x3456);
#pragma unroll
        for (int t = 1; t < 16; ++t) W[t] = __byte_perm(d[t - 1], d[t], 0x3456);
        prev = d[15];
        sha256_compress(st, W, pc);
    }
    // final block: last data byte, 0x80, zeros, 64-bit big-endian bit length
    const uint64_t bits = (uint64_t(leaf) + 1u) * 8u;
    uint32_t W[16];
    W[0] = (prev & 0xff000000u) | 0x00800000u;
#pragma unroll
    for (int t = 1; t < 14; ++t) W[t] = 0u;
    W[14] = uint32_t(bits >> 32);
    W[15] = uint32_t(bits);
    sha256_compress(st, W, pc);
}

// Digest of 0x00 || p[0 .. L) for any L and alignment, byte by byte (the
// short last leaf, or inputs that are not 16-byte aligned).
__device__ void leaf_digest_generic(const uint8_t *__restrict__ p, uint64_t L, uint32_t (&st)[8],
                                    const PipeConst &pc) {
    sha256_init(st);
    const uint64_t ml = L + 1;                 // message bytes
    const uint64_t nblk = (ml + 8) / 64 + 1;   // with 0x80 and the 8-byte length
    const uint64_t len_at = nblk * 64 - 8;
    const uint64_t bits = ml * 8u;
#pragma unroll 1
    for (uint64_t blk = 0; blk < nblk; ++blk) {
        uint32_t W[16];
#pragma unroll 1
        for (int t = 0; t < 16; ++t) {
            uint32_t w = 0;
            for (int j = 0; j < 4; ++j) {
                const uint64_t pos = blk * 64 + 4 * t + j;
                uint32_t byte;
                if (pos == 0) byte = 0x00u;
                else if (pos <= L) byte = p[pos - 1];
                else if (pos == L + 1) byte = 0x80u;
                else if (pos >= len_at) byte = uint32_t(bits >> (56 - 8 * (pos - len_at))) & 0xffu;
                else byte = 0u;
                w = (w << 8) | byte;
            }
            W[t] = w;
        }
        sha256_compress(st, W, pc);
    }
}

// SHA256(0x01 || L || R) for two digests held as big-endian state words.
__device__ __forceinline__ void node_digest(const uint32_t (&L)[8], const uint32_t (&R)[8],
                                            uint32_t (&out)[8], const PipeConst &pc) {
    sha256_init(out);
    uint32_t W[16];
    W[0] = 0x01000000u | (L[0] >> 8);
#pragma unroll
    for (int t = 1; t < 8; ++t) W[t] = (L[t - 1] << 24) | (L[t] >> 8);
    W[8] = (L[7] << 24) | (R[0] >> 8);
#pragma unroll
    for (int t = 9; t < 16; ++t) W[t] = (R[t - 9] << 24) | (R[t - 8] >> 8);
    sha256_compress(out, W, pc);
    // second block: last byte of R, 0x80, zeros, bit length 65 * 8 = 520
    W[0] = (R[7] << 24) | 0x00800000u;
#pragma unroll
    for (int t = 1; t < 15; ++t) W[t] = 0u;
    W[15] = 520u;
    sha256_compress(out, W, pc);
}

__device__ __forceinline__ void store_root(uint8_t *root, const uint32_t (&st)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        root[4 * i] = uint8_t(st[i] >> 24);
        root[4 * i + 1] = uint8_t(st[i] >> 16);
        root[4 * i + 2] = uint8_t(st[i] >> 8);
        root[4 * i + 3] = uint8_t(st[i]);
    }
}

// Optional sink for every node of the tree: level l's nodes are stored in
// index order after all nodes of the levels below it, each as its 32-byte
// digest (big-endian words).  tree == nullptr: nothing is stored.
struct TreeOut {
    uint8_t *tree;
    uint64_t nleaves;
};

// Highest level of a tree of n leaves (the root's level).
__host__ __device__ __forceinline__ int top_level(uint64_t n) {
    int l = 0;
    while (n > 1) { n = (n + 1) / 2; ++l; }
    return l;
}

// Node offset of `level` in the stored tree.
__device__ __forceinline__ uint64_t level_offset(uint64_t n, int level) {
    uint64_t off = 0;
    for (int l = 0; l < level; ++l) { off += n; n = (n + 1) / 2; }
    return off;
}

// The checked build's spans (input bytes, level scratch, root, stored tree)
// and the status word; unused in the release build.
struct MerkleDbg {
    DbgSpan data, ws, root, tree;
    unsigned *status;
};

__device__ __forceinline__ void store_node(const TreeOut &to, int level, uint64_t idx, const uint32_t (&st)[8],
                                           const MerkleDbg &dbg) {
    uint4 *dst = reinterpret_cast<uint4 *>(to.tree + 32 * (level_offset(to.nleaves, level) + idx));
    if (!REPOPS_DBG_OK(dbg.tree, dst, 32, dbg.status)) return;
    dst[0] = make_uint4(__byte_perm(st[0], 0, 0x0123), __byte_perm(st[1], 0, 0x0123),
                        __byte_perm(st[2], 0, 0x0123), __byte_perm(st[3], 0, 0x0123));
    dst[1] = make_uint4(__byte_perm(st[4], 0, 0x0123), __byte_perm(st[5], 0, 0x0123),
                        __byte_perm(st[6], 0, 0x0123), __byte_perm(st[7], 0, 0x0123));
}

// Folds `cnt` digests held word-major in buf[0] ([8][N]) down to buf[?][.][0]
// level by level; returns the buffer index holding the result.  Every thread
// of the CTA must call it (it synchronises).
template <int N>
__device__ __forceinline__ int cta_fold(uint32_t (*buf)[8][N], int cnt, const PipeConst &pc,
                                        const TreeOut &to, int level_in, uint64_t base, int fold_levels,
                                        const MerkleDbg &dbg) {
    int cur = 0;
    int k = 0;   // levels folded so far
    while (cnt > 1) {   // uniform across the CTA
        __syncthreads();
        const int pairs = cnt / 2;
        for (int j = threadIdx.x; j < (cnt + 1) / 2; j += blockDim.x) {
            uint32_t o[8];
            if (j < pairs) {
                uint32_t l[8], r[8];
#pragma unroll
                for (int w = 0; w < 8; ++w) { l[w] = buf[cur][w][2 * j]; r[w] = buf[cur][w][2 * j + 1]; }
                node_digest(l, r, o, pc);
            } else {   // unpaired last node: promoted unchanged
#pragma unroll
                for (int w = 0; w < 8; ++w) o[w] = buf[cur][w][cnt - 1];
            }
#pragma unroll
            for (int w = 0; w < 8; ++w) buf[cur ^ 1][w][j] = o[w];
            if (to.tree) store_node(to, level_in + k + 1, (base >> (k + 1)) + j, o, dbg);
        }
        cur ^= 1;
        cnt = (cnt + 1) / 2;
        ++k;
    }
    __syncthreads();
    // a short block reached one node early: it is promoted through the levels
    // this CTA would still have folded, up to the tree's top
    if (to.tree && threadIdx.x == 0) {
        const int last = min(fold_levels, top_level(to.nleaves) - level_in);
        if (k < last) {
            uint32_t o[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) o[w] = buf[cur][w][0];
            for (int kk = k + 1; kk <= last; ++kk) store_node(to, level_in + kk, base >> kk, o, dbg);
        }
    }
    return cur;
}

__global__ void __launch_bounds__(LEAF_CTA)
// data: the bytes of leaf `first_leaf` onwards (the whole input when 0);
// bytes, nleaves: of the whole input; CTA b folds leaves (cta0 + b) * 128 ..
merkle_leaf_subtree(const uint8_t *__restrict__ data, uint64_t bytes, uint32_t leaf, uint64_t nleaves,
                    int fast_ok, uint32_t *__restrict__ level_out, uint8_t *__restrict__ root_out,
                    const PipeConst pc, const TreeOut to, const MerkleDbg dbg, uint64_t first_leaf,
                    uint64_t cta0) {
    __shared__ uint32_t buf[2][8][LEAF_CTA];
    const uint64_t cta = cta0 + blockIdx.x;
    const uint64_t base = cta * LEAF_CTA;
    const uint64_t i = base + threadIdx.x;
    if (i < nleaves) {
        const uint64_t start = i * leaf;
        const uint64_t len = min(uint64_t(leaf), bytes - start);
        const uint8_t *src = data + (start - first_leaf * leaf);
        uint32_t st[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (REPOPS_DBG_OK(dbg.data, src, uint32_t(len), dbg.status)) {
            if (fast_ok && len == leaf) leaf_digest_fast(src, leaf, st, pc);
            else leaf_digest_generic(src, len, st, pc);
        }
#pragma unroll
        for (int w = 0; w < 8; ++w) buf[0][w][threadIdx.x] = st[w];
        if (to.tree) store_node(to, 0, i, st, dbg);
    }
    const int cnt = int(min(uint64_t(LEAF_CTA), nleaves - base));
    const int cur = cta_fold<LEAF_CTA>(buf, cnt, pc, to, 0, base, LOG_LEAF_CTA, dbg);
    if (threadIdx.x == 0) {
        uint32_t st[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) st[w] = buf[cur][w][0];
        if (root_out) {
            if (REPOPS_DBG_OK(dbg.root, root_out, 32, dbg.status)) store_root(root_out, st);
        } else if (REPOPS_DBG_OK(dbg.ws, level_out + 8 * cta, 32, dbg.status)) {
#pragma unroll
            for (int w = 0; w < 8; ++w) level_out[8 * cta + w] = st[w];
        }
    }
}

__global__ void __launch_bounds__(RED_CTA)
merkle_reduce(const uint32_t *__restrict__ in, uint64_t n, uint32_t *__restrict__ out,
              uint8_t *__restrict__ root_out, const PipeConst pc, const TreeOut to, int level_in,
              const MerkleDbg dbg) {
    __shared__ uint32_t buf[2][8][2 * RED_CTA];
    const uint64_t base = uint64_t(blockIdx.x) * 2 * RED_CTA;
    const int cnt = int(min(uint64_t(2 * RED_CTA), n - base));
    for (int j = threadIdx.x; j < cnt; j += RED_CTA) {
        const bool ok = REPOPS_DBG_OK(dbg.ws, in + 8 * (base + j), 32, dbg.status);
        const uint4 lo = ok ? *reinterpret_cast<const uint4 *>(in + 8 * (base + j)) : make_uint4(0, 0, 0, 0);
        const uint4 hi = ok ? *reinterpret_cast<const uint4 *>(in + 8 * (base + j) + 4) : make_uint4(0, 0, 0, 0);
        buf[0][0][j] = lo.x; buf[0][1][j] = lo.y; buf[0][2][j] = lo.z; buf[0][3][j] = lo.w;
        buf[0][4][j] = hi.x; buf[0][5][j] = hi.y; buf[0][6][j] = hi.z; buf[0][7][j] = hi.w;
    }
    const int cur = cta_fold<2 * RED_CTA>(buf, cnt, pc, to, level_in, base, LOG_RED_NODES, dbg);
    if (threadIdx.x == 0) {
        uint32_t st[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) st[w] = buf[cur][w][0];
        if (root_out) {
            if (REPOPS_DBG_OK(dbg.root, root_out, 32, dbg.status)) store_root(root_out, st);
        } else if (REPOPS_DBG_OK(dbg.ws, out + 8 * blockIdx.x, 32, dbg.status)) {
#pragma unroll
            for (int w = 0; w < 8; ++w) out[8 * blockIdx.x + w] = st[w];
        }
    }
}

struct Plan {
    uint64_t nleaves = 0;
    uint64_t n1 = 0;          // nodes after the leaf kernel
    uint64_t n2 = 0;          // nodes after the first reduce pass
    uint64_t ws_bytes = 0;    // scratch: n1 + n2 nodes of 32 bytes (0 if n1 == 1)
};

bool plan_for(uint64_t bytes, uint32_t leaf, Plan *p) {
    if (bytes == 0 || leaf < 64 || leaf % 64 != 0 || leaf > (1u << 30)) return false;
    p->nleaves = (bytes + leaf - 1) / leaf;
    p->n1 = (p->nleaves + LEAF_CTA - 1) / LEAF_CTA;
    if (p->n1 > 0x7fffffffull) return false;
    p->n2 = p->n1 > 1 ? (p->n1 + 2 * RED_CTA - 1) / (2 * RED_CTA) : 0;
    p->ws_bytes = p->n1 > 1 ? (p->n1 + p->n2) * 32u : 0;
    return true;
}

uint64_t total_nodes(uint64_t nleaves);
int reduce_levels(const Plan &pl, uint8_t *root_out, uint32_t *bufA, uint32_t *bufB, const PipeConst &pc,
                  const TreeOut &to, const MerkleDbg &dbg, cudaStream_t stream);

int run(const void *ptr, uint64_t bytes, uint32_t leaf, uint8_t *root_out, void *ws, const Plan &pl,
        cudaStream_t stream, const TreeOut to = TreeOut{nullptr, 0}) {
    const uint8_t *data = static_cast<const uint8_t *>(ptr);
    const int fast_ok = reinterpret_cast<uintptr_t>(data) % 16 == 0;
    const PipeConst pc{1u};
    uint32_t *bufA = static_cast<uint32_t *>(ws);
    uint32_t *bufB = bufA ? bufA + 8 * pl.n1 : nullptr;
    MerkleDbg dbg{};
    dbg.data = dbg_span(data, bytes);
    dbg.ws = dbg_span(ws, pl.ws_bytes);
    dbg.root = dbg_span(root_out, 32);
    dbg.tree = dbg_span(to.tree, to.tree ? total_nodes(to.nleaves) * 32u : 0);
    int rc = status_word_address(&dbg.status);
    if (rc != REPOPS_OK) return rc;
    merkle_leaf_subtree<<<unsigned(pl.n1), LEAF_CTA, 0, stream>>>(
        data, bytes, leaf, pl.nleaves, fast_ok, bufA, pl.n1 == 1 ? root_out : nullptr, pc, to, dbg, 0, 0);
    rc = check_launch();
    if (rc != REPOPS_OK) return rc;
    return reduce_levels(pl, root_out, bufA, bufB, pc, to, dbg, stream);
}

// The reduce passes over the leaf kernel's level-7 nodes in bufA (bufB the
// other half of the scratch), down to the root.
int reduce_levels(const Plan &pl, uint8_t *root_out, uint32_t *bufA, uint32_t *bufB, const PipeConst &pc,
                  const TreeOut &to, const MerkleDbg &dbg, cudaStream_t stream) {
    int rc = REPOPS_OK;
    uint64_t n = pl.n1;
    int level = LOG_LEAF_CTA;
    uint32_t *src = bufA, *dst = bufB;
    while (n > 1) {
        const uint64_t blocks = (n + 2 * RED_CTA - 1) / (2 * RED_CTA);
        merkle_reduce<<<unsigned(blocks), RED_CTA, 0, stream>>>(src, n, dst, blocks == 1 ? root_out : nullptr,
                                                                pc, to, level, dbg);
        rc = check_launch();
        if (rc != REPOPS_OK) return rc;
        n = blocks;
        level += LOG_RED_NODES;
        std::swap(src, dst);
    }
    return REPOPS_OK;
}

int check_args(const void *ptr, uint64_t bytes, uint32_t leaf, const uint8_t *root_out, Plan *pl) {
    if (!ptr || !root_out) return REPOPS_ERR_INVALID_ARG;
    if (!plan_for(bytes, leaf, pl)) return REPOPS_ERR_INVALID_ARG;
    if (ranges_overlap(ptr, bytes, root_out, 32)) return REPOPS_ERR_ALIAS;
    return REPOPS_OK;
}

}  // namespace
}  // namespace repops

using namespace repops;

extern "C" uint64_t repops_merkle_workspace_bytes(uint64_t bytes, uint32_t leaf) {
    Plan pl;
    return plan_for(bytes, leaf, &pl) ? pl.ws_bytes : 0;
}

extern "C" int repops_merkle_sha256_ws(const void *ptr, uint64_t bytes, uint32_t leaf, uint8_t *root_out,
                                       void *workspace, uint64_t workspace_bytes, cudaStream_t stream) {
    Plan pl;
    int rc = check_args(ptr, bytes, leaf, root_out, &pl);
    if (rc != REPOPS_OK) return rc;
    if (pl.ws_bytes > 0) {
        if (!workspace || workspace_bytes < pl.ws_bytes || reinterpret_cast<uintptr_t>(workspace) % 16)
            return REPOPS_ERR_INVALID_ARG;
        if (ranges_overlap(workspace, pl.ws_bytes, ptr, bytes) ||
            ranges_overlap(workspace, pl.ws_bytes, root_out, 32))
            return REPOPS_ERR_ALIAS;
    }
    return run(ptr, bytes, leaf, root_out, pl.ws_bytes ? workspace : nullptr, pl, stream);
}

extern "C" int repops_merkle_sha256(const void *ptr, uint64_t bytes, uint32_t leaf, uint8_t *root_out,
                                    cudaStream_t stream) {
    Plan pl;
    int rc = check_args(ptr, bytes, leaf, root_out, &pl);
    if (rc != REPOPS_OK) return rc;
    void *ws = nullptr;
    if (pl.ws_bytes > 0) {
        cudaError_t e = scratch_malloc(&ws, pl.ws_bytes, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return REPOPS_ERR_ALLOC;
        }
    }
    rc = run(ptr, bytes, leaf, root_out, ws, pl, stream);
    if (ws) {
        cudaError_t e = cudaFreeAsync(ws, stream);
        if (e != cudaSuccess && rc == REPOPS_OK) rc = set_cuda_error(e);
    }
    return rc;
}

// ---------------------------------------------------------------------------
// Whole tree, inclusion proofs, verification ("Verde与RepOps" §2.4: the
// referee asks for a Merkle membership proof of an input tensor hash against
// the checkpoint).  A proof is the list of sibling digests on the path from a
// leaf to the root, bottom-up, one per level where the path's node has a
// sibling; its shape follows from (leaf count, leaf index) alone.
// ---------------------------------------------------------------------------

namespace repops {
namespace {

__host__ __device__ __forceinline__ int path_steps(uint64_t nleaves, uint64_t index) {
    int steps = 0;
    uint64_t count = nleaves, j = index;
    while (count > 1) {
        if ((j & 1) || j + 1 < count) ++steps;
        count = (count + 1) / 2;
        j >>= 1;
    }
    return steps;
}

__device__ __forceinline__ void load_digest(const uint8_t *p, uint32_t (&w)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = (uint32_t(p[4 * i]) << 24) | (uint32_t(p[4 * i + 1]) << 16) | (uint32_t(p[4 * i + 2]) << 8) |
               uint32_t(p[4 * i + 3]);
}

// One thread gathers the siblings of leaf `index` from the stored tree.
__global__ void merkle_proof_kernel(const uint8_t *__restrict__ tree, uint64_t nleaves, uint64_t index,
                                    uint8_t *__restrict__ proof) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    uint64_t off = 0, count = nleaves, j = index;
    int s = 0;
    while (count > 1) {
        uint64_t sib = 0;
        bool has = true;
        if (j & 1) sib = j - 1;
        else if (j + 1 < count) sib = j + 1;
        else has = false;
        if (has) {
            const uint8_t *src = tree + 32 * (off + sib);
            for (int b = 0; b < 32; ++b) proof[32 * s + b] = src[b];
            ++s;
        }
        off += count;
        count = (count + 1) / 2;
        j >>= 1;
    }
}

// One thread hashes the leaf bytes, climbs with the siblings and compares the
// result with the root: *ok = 1 (member) or 0.
__global__ void merkle_verify_kernel(const uint8_t *__restrict__ leaf_bytes, uint64_t leaf_len,
                                     uint64_t nleaves, uint64_t index, const uint8_t *__restrict__ proof,
                                     const uint8_t *__restrict__ root, int *__restrict__ ok,
                                     const PipeConst pc) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    uint32_t h[8];
    leaf_digest_generic(leaf_bytes, leaf_len, h, pc);
    uint64_t count = nleaves, j = index;
    int s = 0;
    while (count > 1) {
        const bool left_sib = (j & 1) != 0, right_sib = !(j & 1) && j + 1 < count;
        if (left_sib || right_sib) {
            uint32_t sib[8], o[8];
            load_digest(proof + 32 * s, sib);
            ++s;
            if (left_sib) node_digest(sib, h, o, pc);
            else node_digest(h, sib, o, pc);
#pragma unroll
            for (int w = 0; w < 8; ++w) h[w] = o[w];
        }
        count = (count + 1) / 2;
        j >>= 1;
    }
    uint32_t r[8];
    load_digest(root, r);
    bool same = true;
#pragma unroll
    for (int w = 0; w < 8; ++w) same = same && (r[w] == h[w]);
    *ok = same ? 1 : 0;
}

uint64_t total_nodes(uint64_t nleaves) {
    uint64_t t = 0, c = nleaves;
    for (;;) {
        t += c;
        if (c == 1) break;
        c = (c + 1) / 2;
    }
    return t;
}

}  // namespace
}  // namespace repops

extern "C" uint64_t repops_merkle_tree_bytes(uint64_t bytes, uint32_t leaf) {
    Plan pl;
    if (!plan_for(bytes, leaf, &pl)) return 0;
    return 32 * total_nodes(pl.nleaves);
}

namespace repops {
namespace {

// Streams and events of one host-buffer call, destroyed (deferred by the
// runtime until their work completes) when the call returns.
struct HostMerkleRes {
    cudaStream_t in = nullptr;
    cudaEvent_t ev[4] = {};
    ~HostMerkleRes() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);
        if (in) cudaStreamDestroy(in);
    }
};

}  // namespace
}  // namespace repops

extern "C" int repops_merkle_sha256_host(const void *ptr, uint64_t bytes, uint32_t leaf, uint8_t *root_out,
                                         cudaStream_t stream) {
    Plan pl;
    int rc = check_args(ptr, bytes, leaf, root_out, &pl);
    if (rc != REPOPS_OK) return rc;
    // chunks of whole 128-leaf CTAs, about 64 MiB each, double-buffered
    const uint64_t cta_bytes = uint64_t(LEAF_CTA) * leaf;
    const uint64_t per_chunk = std::max<uint64_t>(1, (uint64_t(64) << 20) / cta_bytes);
    const uint64_t chunk_bytes = std::min<uint64_t>(per_chunk * cta_bytes, (bytes + cta_bytes - 1) / cta_bytes * cta_bytes);
    const uint64_t nchunks = (bytes + chunk_bytes - 1) / chunk_bytes;
    const uint64_t ws_bytes = (pl.ws_bytes + 255) / 256 * 256;
    void *mem = nullptr;
    if (scratch_malloc(&mem, ws_bytes + 2 * chunk_bytes + 256, stream) != cudaSuccess) {
        cudaGetLastError();
        return REPOPS_ERR_ALLOC;
    }
    unsigned char *base = static_cast<unsigned char *>(mem);
    uint32_t *bufA = pl.ws_bytes ? reinterpret_cast<uint32_t *>(base) : nullptr;
    uint32_t *bufB = bufA ? bufA + 8 * pl.n1 : nullptr;
    uint8_t *chunk[2] = {base + ws_bytes, base + ws_bytes + chunk_bytes};
    uint8_t *droot = base + ws_bytes + 2 * chunk_bytes;
    HostMerkleRes res;
    cudaError_t e = cudaStreamCreateWithFlags(&res.in, cudaStreamNonBlocking);
    for (int k = 0; k < 4 && e == cudaSuccess; ++k) e = cudaEventCreateWithFlags(&res.ev[k], cudaEventDisableTiming);
    // ev[0]: the allocation is ordered; ev[1 + b]: chunk buffer b's bytes are in;
    // ev[3]: reused per chunk for "the leaf kernel of the previous use of a
    // buffer is done" (recorded on `stream`, waited on by `in`)
    if (e == cudaSuccess) e = cudaEventRecord(res.ev[0], stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(res.in, res.ev[0], 0);
    const PipeConst pc{1u};
    MerkleDbg dbg{};
    dbg.ws = dbg_span(bufA, pl.ws_bytes);
    dbg.root = dbg_span(droot, 32);
    if (e == cudaSuccess) rc = status_word_address(&dbg.status);
    cudaEvent_t done[2] = {nullptr, nullptr};
    for (uint64_t c = 0; e == cudaSuccess && rc == REPOPS_OK && c < nchunks; ++c) {
        const int b = int(c & 1);
        const uint64_t off = c * chunk_bytes, cb = std::min(chunk_bytes, bytes - off);
        if (done[b] && (e = cudaStreamWaitEvent(res.in, done[b], 0)) != cudaSuccess) break;
        if ((e = cudaMemcpyAsync(chunk[b], static_cast<const uint8_t *>(ptr) + off, cb, cudaMemcpyHostToDevice,
                                 res.in)) != cudaSuccess ||
            (e = cudaEventRecord(res.ev[1 + b], res.in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(stream, res.ev[1 + b], 0)) != cudaSuccess)
            break;
        const uint64_t first_leaf = off / leaf, leaves = (cb + leaf - 1) / leaf;
        const uint64_t ctas = (leaves + LEAF_CTA - 1) / LEAF_CTA;
        dbg.data = dbg_span(chunk[b], cb);
        merkle_leaf_subtree<<<unsigned(ctas), LEAF_CTA, 0, stream>>>(
            chunk[b], bytes, leaf, pl.nleaves, 1, bufA, pl.n1 == 1 ? droot : nullptr, pc, TreeOut{nullptr, 0}, dbg,
            first_leaf, off / cta_bytes);
        rc = check_launch();
        if (rc != REPOPS_OK) break;
        // the buffer is free again once this leaf kernel is done
        cudaEvent_t ev = nullptr;
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) break;
        e = cudaEventRecord(ev, stream);
        if (done[b]) cudaEventDestroy(done[b]);
        done[b] = ev;
    }
    for (cudaEvent_t d : done)
        if (d) cudaEventDestroy(d);
    if (rc == REPOPS_OK && e == cudaSuccess && pl.n1 > 1)
        rc = reduce_levels(pl, droot, bufA, bufB, pc, TreeOut{nullptr, 0}, dbg, stream);
    if (rc == REPOPS_OK && e == cudaSuccess)
        e = cudaMemcpyAsync(root_out, droot, 32, cudaMemcpyDeviceToHost, stream);
    // every copy into the chunk buffers is over before they are released, also
    // when an error stopped the loop half-way
    const cudaError_t j = join_helper_streams(stream, res.in, nullptr);
    if (e == cudaSuccess) e = j;
    const cudaError_t f = cudaFreeAsync(mem, stream);
    if (rc != REPOPS_OK) return rc;
    if (e != cudaSuccess) return set_cuda_error(e);
    if (f != cudaSuccess) return set_cuda_error(f);
    return REPOPS_OK;
}

extern "C" int repops_merkle_tree_sha256(const void *ptr, uint64_t bytes, uint32_t leaf, uint8_t *tree,
                                         uint64_t tree_bytes, uint8_t *root_out, cudaStream_t stream) {
    Plan pl;
    int rc = check_args(ptr, bytes, leaf, root_out, &pl);
    if (rc != REPOPS_OK) return rc;
    const uint64_t need = 32 * total_nodes(pl.nleaves);
    if (!tree || tree_bytes < need || reinterpret_cast<uintptr_t>(tree) % 16) return REPOPS_ERR_INVALID_ARG;
    if (ranges_overlap(tree, need, ptr, bytes) || ranges_overlap(tree, need, root_out, 32)) return REPOPS_ERR_ALIAS;
    void *ws = nullptr;
    if (pl.ws_bytes > 0) {
        cudaError_t e = scratch_malloc(&ws, pl.ws_bytes, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return REPOPS_ERR_ALLOC;
        }
    }
    rc = run(ptr, bytes, leaf, root_out, ws, pl, stream, TreeOut{tree, pl.nleaves});
    if (ws) {
        cudaError_t e = cudaFreeAsync(ws, stream);
        if (e != cudaSuccess && rc == REPOPS_OK) rc = set_cuda_error(e);
    }
    return rc;
}

extern "C" int repops_merkle_proof_steps(uint64_t nleaves, uint64_t index) {
    if (nleaves == 0 || index >= nleaves) return REPOPS_ERR_INVALID_ARG;
    return path_steps(nleaves, index);
}

extern "C" int repops_merkle_proof(const uint8_t *tree, uint64_t nleaves, uint64_t index, uint8_t *proof_out,
                                   cudaStream_t stream) {
    if (!tree || !proof_out || nleaves == 0 || index >= nleaves) return REPOPS_ERR_INVALID_ARG;
    const uint64_t tree_bytes = 32 * total_nodes(nleaves);
    if (ranges_overlap(tree, tree_bytes, proof_out, 32u * uint64_t(path_steps(nleaves, index))))
        return REPOPS_ERR_ALIAS;
    merkle_proof_kernel<<<1, 32, 0, stream>>>(tree, nleaves, index, proof_out);
    return check_launch();
}

extern "C" int repops_merkle_verify(const void *leaf_bytes, uint64_t leaf_len, uint64_t nleaves, uint64_t index,
                                    const uint8_t *proof, const uint8_t *root, int *ok_out, cudaStream_t stream) {
    if ((!leaf_bytes && leaf_len) || !root || !ok_out || nleaves == 0 || index >= nleaves)
        return REPOPS_ERR_INVALID_ARG;
    if (!proof && path_steps(nleaves, index) > 0) return REPOPS_ERR_INVALID_ARG;
    const PipeConst pc{1u};
    merkle_verify_kernel<<<1, 32, 0, stream>>>(static_cast<const uint8_t *>(leaf_bytes), leaf_len, nleaves, index,
                                               proof, root, ok_out, pc);
    return check_launch();
}

// ---------------------------------------------------------------------------
// Compression-rate probe: the same compression with its message in registers,
// no loads and no tree, as the ceiling the Merkle kernels are measured
// against.  Thread t hashes the message M_t^iters (M_t = the 16 big-endian
// words 16t, 16t + 1, ..., 16t + 15, repeated iters times) and writes its
// SHA-256 digest as 8 words.
// ---------------------------------------------------------------------------

namespace repops {
namespace {

__global__ void __launch_bounds__(LEAF_CTA)
sha256_rate_kernel(uint32_t iters, uint32_t *__restrict__ out, const PipeConst pc) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t st[8];
    sha256_init(st);
#pragma unroll 1
    for (uint32_t r = 0; r < iters; ++r) {
        uint32_t W[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) W[i] = 16u * t + uint32_t(i);
        sha256_compress(st, W, pc);
    }
    const uint64_t bits = uint64_t(iters) * 512u;
    uint32_t W[16];
    W[0] = 0x80000000u;
#pragma unroll
    for (int i = 1; i < 14; ++i) W[i] = 0u;
    W[14] = uint32_t(bits >> 32);
    W[15] = uint32_t(bits);
    sha256_compress(st, W, pc);
#pragma unroll
    for (int w = 0; w < 8; ++w) out[8 * uint64_t(t) + w] = st[w];
}

}  // namespace
}  // namespace repops

extern "C" int repops_sha256_rate_probe(uint32_t threads, uint32_t iters, uint32_t *digests, cudaStream_t stream) {
    using namespace repops;
    if (!digests || threads == 0 || threads % LEAF_CTA != 0 || threads > (1u << 24) || iters > (1u << 30))
        return REPOPS_ERR_INVALID_ARG;
    const PipeConst pc{1u};
    sha256_rate_kernel<<<threads / LEAF_CTA, LEAF_CTA, 0, stream>>>(iters, digests, pc);
    return check_launch();
}

// ---------------------------------------------------------------------------
// Allocation-free variant.
//
// For callers that must not allocate device memory when they hash: a host
// framework that has reserved all device memory for its own pool, a
// latency-critical path on which an allocation could block or synchronise, or
// a plug-in whose host forbids allocations after start-up.  The scratch of the
// level nodes lives in the fixed array below instead of coming from the
// library's scratch pool or from the caller.
//
// The array is part of the library's device image: every GPU that loads the
// library holds these bytes until the process exits.  All calls share it and
// it keeps whatever the last call left there; nothing in it needs to start at
// zero, because every node is written before it is read.  Two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array and may return wrong roots.
// ---------------------------------------------------------------------------

static_assert(REPOPS_MERKLE_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");
static __device__ __align__(256) unsigned char g_merkle_noalloc_scratch[REPOPS_MERKLE_NOALLOC_SCRATCH_BYTES];

namespace repops {
namespace {

constexpr int kNoallocMaxDevices = 64;

// Device address of the scratch array, looked up once per device and context
// with that device current.  In host code the array's name only stands in for
// the symbol; its device address is valid in the context it was looked up in
// only, so a new context on the device (after cudaDeviceReset, say) looks it
// up again instead of reusing a stale address.
struct NoallocAddr {
    std::mutex mu;
    uint64_t ctx_key = 0;
    void *addr = nullptr;
};
NoallocAddr g_noalloc_scratch_addr[kNoallocMaxDevices];

int noalloc_scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev < 0 || dev >= kNoallocMaxDevices) return REPOPS_ERR_UNSUPPORTED;
    uint64_t key = 0;
    int rc = current_context_key(&key);
    if (rc != REPOPS_OK) return rc;
    NoallocAddr &a = g_noalloc_scratch_addr[dev];
    std::lock_guard<std::mutex> lock(a.mu);
    if (a.ctx_key != key || !a.addr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_merkle_noalloc_scratch);
        if (e != cudaSuccess) return set_cuda_error(e);
        a.addr = p;
        a.ctx_key = key;
    }
    *out = a.addr;
    return REPOPS_OK;
}

}  // namespace
}  // namespace repops

extern "C" int repops_merkle_sha256_noalloc(const void *ptr, uint64_t bytes, uint32_t leaf,
                                            uint8_t *root_out, cudaStream_t stream) {
    Plan pl;
    int rc = check_args(ptr, bytes, leaf, root_out, &pl);
    if (rc != REPOPS_OK) return rc;
    if (pl.ws_bytes > REPOPS_MERKLE_NOALLOC_SCRATCH_BYTES) return REPOPS_ERR_UNSUPPORTED;
    void *ws = nullptr;
    if (pl.ws_bytes > 0) {
        rc = noalloc_scratch_address(&ws);
        if (rc != REPOPS_OK) return rc;
    }
    return run(ptr, bytes, leaf, root_out, ws, pl, stream);
}
