/*
 * repops_oracle.c -- the CPU oracle for the reproducible-operator hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * statement of what the GPU library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it.  It shares no source,
 * header, table or constant with the CUDA library, and never calls it.
 *
 * Build flags (oracle/build.py): -std=c11 -O2 -ffp-contract=off -fno-fast-math.
 * -ffp-contract=off matters: GCC's default in GNU mode would fuse a*b+c into a
 * fused multiply-add on aarch64, which is exactly what the method forbids.
 *
 * Sources (page title, section):
 *  [RepOps]  "Verde与RepOps：机器学习可验证委托与硬件无关确定性",
 *            §3.1 (sources of non-determinism), §3.2 (design principle and the
 *            matmul example: any order over i and j, fixed order over k,
 *            sum starts at 0, sum = sum + a*b), §3.3 (IEEE-754 requirement),
 *            §2.3.2 (checkpoint hash is a Merkle tree over node hashes),
 *            §2.4 (Merkle membership proof of an input tensor hash).
 *  [Zoo]     "Zoo Per-LLM Chain Soundness", §2 Definition "Aggregation rule",
 *            Lemma "Order independence within a batch"; §5 "Detailed proof:
 *            deterministic ordering", paragraphs "Ordering subroutine",
 *            "Determinism of left-fold" (round-to-nearest-even, FMA off) and
 *            "Update step"; §1 "Background" (batch hash = Merkle root);
 *            §6 table "Per-LLM chain block field layout" (bytes32 roots);
 *            §7 "Reproducibility test plan" (verify H(theta) = m).
 *  [FIPS]    FIPS PUB 180-4, Secure Hash Standard: SHA-256 (§4.1.2 functions,
 *            §4.2.2 constants, §5.1.1 padding, §5.3.3 initial value,
 *            §6.2 computation).
 *
 * Readings taken where the pages are silent:
 *  - no FMA: the product is rounded to binary32, then added with its own
 *    rounding; rounding is to nearest even; subnormals are kept (no FTZ/DAZ);
 *  - the GEMM sum starts at +0.0f;
 *  - the contributor mean starts the left fold at the first sorted gradient,
 *    then divides by |C| with one correctly rounded division;
 *  - SGD: theta = theta - (eta * gbar), each op rounded;
 *  - the hash is SHA-256; leaf = SHA256(0x00 || leaf bytes), node =
 *    SHA256(0x01 || left || right); leaves cut from the tensor bytes in
 *    increasing offset, the last one possibly short; level by level, pairs
 *    (0,1),(2,3),...; an unpaired last node is promoted unchanged;
 *  - a GEMM epilogue runs after the whole k-chain of its element:
 *    y = alpha*acc, then + bias[j], then GeLU, then + residual, each rounded.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>   /* rintf, rint, sqrtf: IEEE round-to-integral and correctly rounded square root */

/* ------------------------------------------------------------------------ */
/* Floating-point environment                                                */
/* ------------------------------------------------------------------------ */

/* Returns 1 when the host keeps subnormal results and subnormal inputs
 * (no flush-to-zero, no denormals-are-zero) and rounds to nearest even.
 * [RepOps §3.3] needs IEEE-754 behaviour; [Zoo §5] pins round-to-nearest-even. */
int oracle_fp_env_ok(void)
{
    volatile float tiny = 1.17549435e-38f;      /* FLT_MIN, smallest normal */
    volatile float half = 0.5f;
    volatile float sub = tiny * half;           /* 2^-127: subnormal */
    if (sub == 0.0f) return 0;                  /* FTZ on outputs */
    volatile float sub2 = sub + 0.0f;
    if (sub2 == 0.0f) return 0;                 /* DAZ on inputs */
    /* ties-to-even: 1 + 2^-24 is exactly half-way between 1 and 1 + 2^-23 */
    volatile float one = 1.0f;
    volatile float h = 5.9604644775390625e-08f; /* 2^-24 */
    volatile float t = one + h;
    if (t != 1.0f) return 0;
    volatile float odd = 1.00000011920928955078125f; /* 1 + 2^-23 */
    volatile float t2 = odd + h;                     /* tie: goes to 1 + 2^-22 */
    if (t2 != 1.0000002384185791015625f) return 0;
    return 1;
}

/* ------------------------------------------------------------------------ */
/* Order-fixed GEMM  [RepOps §3.2, matmul example]                           */
/* ------------------------------------------------------------------------ */

/* C[i][j] = ((0 + A[i][0]*B[0][j]) + A[i][1]*B[1][j]) + ... + A[i][K-1]*B[K-1][j]
 * with every product and every sum rounded to binary32.
 *
 * Storage: row-major with leading dimensions in elements.
 *   transA == 0: A(i,k) = A[i*lda + k]      transA != 0: A(i,k) = A[k*lda + i]
 *   transB == 0: B(k,j) = B[k*ldb + j]      transB != 0: B(k,j) = B[j*ldb + k]
 *   C(i,j) = C[i*ldc + j]
 * The loops follow the page: i and j in any order (here increasing), k in
 * strictly increasing order. */
void oracle_gemm_f32(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda, int transA,
                     const float *B, int64_t ldb, int transB,
                     float *C, int64_t ldc)
{
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            float sum = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float a = transA ? A[k * lda + i] : A[i * lda + k];
                float b = transB ? B[j * ldb + k] : B[k * ldb + j];
                float p = a * b;        /* product, rounded to binary32 */
                sum = sum + p;          /* sum, rounded to binary32     */
            }
            C[i * ldc + j] = sum;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Contributor order  [Zoo §2 Lemma "Order independence"; §5 "Ordering       */
/* subroutine"; §6 "contributors (sorted DID list)"]                         */
/* ------------------------------------------------------------------------ */

/* Lexicographic comparison on unsigned bytes; a proper prefix sorts first. */
static int id_less(const uint8_t *a, int64_t la, const uint8_t *b, int64_t lb)
{
    int64_t n = la < lb ? la : lb;
    for (int64_t i = 0; i < n; ++i) {
        if (a[i] != b[i]) return a[i] < b[i];
    }
    return la < lb;
}

/* ids: concatenated identifier bytes; offs[r], lens[r]: where contributor r's
 * identifier starts and how long it is.  Writes order[0..n-1] such that
 * order[0] is the contributor with the smallest identifier.  Returns 0, or -1
 * if two identifiers are equal (the contributor set would not be a set). */
int oracle_sort_ids(int n, const uint8_t *ids, const int64_t *offs,
                    const int64_t *lens, int *order)
{
    for (int r = 0; r < n; ++r) order[r] = r;
    /* insertion sort: plain and stable */
    for (int r = 1; r < n; ++r) {
        int cur = order[r];
        int s = r - 1;
        while (s >= 0 && id_less(ids + offs[cur], lens[cur],
                                 ids + offs[order[s]], lens[order[s]])) {
            order[s + 1] = order[s];
            --s;
        }
        order[s + 1] = cur;
    }
    for (int r = 1; r < n; ++r) {
        const int p = order[r - 1], q = order[r];
        if (!id_less(ids + offs[p], lens[p], ids + offs[q], lens[q])) return -1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Fixed-order contributor mean fused with SGD                               */
/* [Zoo §2 Def. "Aggregation rule"; §5 "Ordering subroutine" (left fold),    */
/*  "Update step" (theta_t = theta_{t-1} - eta * gbar_t)]                    */
/* ------------------------------------------------------------------------ */

/* For each element e:
 *   S = g[order[0]][e];  S = S + g[order[r]][e] for r = 1..nC-1  (left fold)
 *   gbar = S / nC                       (one correctly rounded division)
 *   theta[e] = theta[e] - (eta * gbar)  (product rounded, then difference)
 * Returns 0, or -1 if order is not a permutation of 0..nC-1 or nC < 1. */
int oracle_mean_sgd(int nC, int64_t len, const float *const *grads,
                    const int *order, float eta, float *theta)
{
    if (nC < 1) return -1;
    char *seen = (char *)calloc((size_t)nC, 1);
    if (!seen) return -1;
    for (int r = 0; r < nC; ++r) {
        if (order[r] < 0 || order[r] >= nC || seen[order[r]]) { free(seen); return -1; }
        seen[order[r]] = 1;
    }
    free(seen);
    const float count = (float)nC;   /* exact for nC < 2^24 */
    for (int64_t e = 0; e < len; ++e) {
        float S = grads[order[0]][e];
        for (int r = 1; r < nC; ++r) {
            S = S + grads[order[r]][e];
        }
        float gbar = S / count;
        float step = eta * gbar;
        theta[e] = theta[e] - step;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* SHA-256  [FIPS 180-4]                                                     */
/* ------------------------------------------------------------------------ */

static uint32_t sha_K[64];
static uint32_t sha_H0[8];
static int sha_ready = 0;

/* floor(cbrt(v)) for v < 2^120, by bisection on exact integers. */
static uint64_t icbrt128(unsigned __int128 v)
{
    uint64_t lo = 0, hi = (uint64_t)1 << 41;   /* hi^3 = 2^123 > v */
    while (hi - lo > 1) {
        uint64_t mid = lo + (hi - lo) / 2;
        unsigned __int128 m = mid;
        if (m * m * m <= v) lo = mid; else hi = mid;
    }
    return lo;
}

/* floor(sqrt(v)) for v < 2^120. */
static uint64_t isqrt128(unsigned __int128 v)
{
    uint64_t lo = 0, hi = (uint64_t)1 << 61;   /* hi^2 = 2^122 > v */
    while (hi - lo > 1) {
        uint64_t mid = lo + (hi - lo) / 2;
        unsigned __int128 m = mid;
        if (m * m <= v) lo = mid; else hi = mid;
    }
    return lo;
}

/* FIPS 180-4 §4.2.2: K[t] is the first 32 bits of the fractional part of the
 * cube root of the t-th prime; §5.3.3: H0[i] the first 32 bits of the
 * fractional part of the square root of the i-th prime.  Derived here in exact
 * integer arithmetic: floor(cbrt(p) * 2^32) = floor(cbrt(p * 2^96)), and its
 * low 32 bits drop the integer part. */
static void sha_init_constants(void)
{
    if (sha_ready) return;
    int primes[64];
    int count = 0;
    for (int c = 2; count < 64; ++c) {
        int is_prime = 1;
        for (int d = 2; d * d <= c; ++d) {
            if (c % d == 0) { is_prime = 0; break; }
        }
        if (is_prime) primes[count++] = c;
    }
    for (int t = 0; t < 64; ++t) {
        unsigned __int128 v = (unsigned __int128)primes[t] << 96;
        sha_K[t] = (uint32_t)(icbrt128(v) & 0xffffffffu);
    }
    for (int i = 0; i < 8; ++i) {
        unsigned __int128 v = (unsigned __int128)primes[i] << 64;
        sha_H0[i] = (uint32_t)(isqrt128(v) & 0xffffffffu);
    }
    sha_ready = 1;
}

void oracle_sha256_constants(uint32_t K_out[64], uint32_t H0_out[8])
{
    sha_init_constants();
    memcpy(K_out, sha_K, sizeof(sha_K));
    memcpy(H0_out, sha_H0, sizeof(sha_H0));
}

static uint32_t rotr32(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

/* FIPS 180-4 §6.2.2: process one 512-bit block. */
static void sha_block(uint32_t H[8], const uint8_t blk[64])
{
    uint32_t W[64];
    for (int t = 0; t < 16; ++t) {
        W[t] = ((uint32_t)blk[4 * t] << 24) | ((uint32_t)blk[4 * t + 1] << 16) |
               ((uint32_t)blk[4 * t + 2] << 8) | (uint32_t)blk[4 * t + 3];
    }
    for (int t = 16; t < 64; ++t) {
        uint32_t s0 = rotr32(W[t - 15], 7) ^ rotr32(W[t - 15], 18) ^ (W[t - 15] >> 3);
        uint32_t s1 = rotr32(W[t - 2], 17) ^ rotr32(W[t - 2], 19) ^ (W[t - 2] >> 10);
        W[t] = s1 + W[t - 7] + s0 + W[t - 16];
    }
    uint32_t a = H[0], b = H[1], c = H[2], d = H[3];
    uint32_t e = H[4], f = H[5], g = H[6], h = H[7];
    for (int t = 0; t < 64; ++t) {
        uint32_t S1 = rotr32(e, 6) ^ rotr32(e, 11) ^ rotr32(e, 25);
        uint32_t ch = (e & f) ^ (~e & g);
        uint32_t T1 = h + S1 + ch + sha_K[t] + W[t];
        uint32_t S0 = rotr32(a, 2) ^ rotr32(a, 13) ^ rotr32(a, 22);
        uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
        uint32_t T2 = S0 + maj;
        h = g; g = f; f = e; e = d + T1;
        d = c; c = b; b = a; a = T1 + T2;
    }
    H[0] += a; H[1] += b; H[2] += c; H[3] += d;
    H[4] += e; H[5] += f; H[6] += g; H[7] += h;
}

typedef struct {
    uint32_t H[8];
    uint64_t total;     /* message bytes consumed so far */
    uint8_t buf[64];
    unsigned fill;
} osha_ctx;

static void osha_init(osha_ctx *c)
{
    sha_init_constants();
    memcpy(c->H, sha_H0, sizeof(sha_H0));
    c->total = 0;
    c->fill = 0;
}

static void osha_update(osha_ctx *c, const uint8_t *p, uint64_t n)
{
    c->total += n;
    while (n > 0) {
        unsigned take = 64 - c->fill;
        if ((uint64_t)take > n) take = (unsigned)n;
        memcpy(c->buf + c->fill, p, take);
        c->fill += take;
        p += take;
        n -= take;
        if (c->fill == 64) {
            sha_block(c->H, c->buf);
            c->fill = 0;
        }
    }
}

/* FIPS 180-4 §5.1.1: append 0x80, zeros, and the 64-bit big-endian bit length. */
static void osha_final(osha_ctx *c, uint8_t out[32])
{
    uint64_t bits = c->total * 8u;
    uint8_t one = 0x80, zero = 0;
    uint64_t keep_total = c->total;
    osha_update(c, &one, 1);
    while (c->fill != 56) osha_update(c, &zero, 1);
    uint8_t len[8];
    for (int i = 0; i < 8; ++i) len[i] = (uint8_t)(bits >> (56 - 8 * i));
    osha_update(c, len, 8);
    c->total = keep_total;
    for (int i = 0; i < 8; ++i) {
        out[4 * i] = (uint8_t)(c->H[i] >> 24);
        out[4 * i + 1] = (uint8_t)(c->H[i] >> 16);
        out[4 * i + 2] = (uint8_t)(c->H[i] >> 8);
        out[4 * i + 3] = (uint8_t)(c->H[i]);
    }
}

void oracle_sha256(const uint8_t *msg, uint64_t len, uint8_t out[32])
{
    osha_ctx c;
    osha_init(&c);
    osha_update(&c, msg, len);
    osha_final(&c, out);
}

/* ------------------------------------------------------------------------ */
/* Merkle commitment over tensor bytes                                       */
/* [Zoo §1 "batch hash (Merkle root over input batch)", §6 bytes32 roots,    */
/*  §7 "verify H(theta) = m"; RepOps §2.3.2 Merkle tree over node hashes]    */
/* ------------------------------------------------------------------------ */

/* Leaf i covers bytes [i*leaf, min((i+1)*leaf, n)):  SHA256(0x00 || bytes). */
static void merkle_leaf(const uint8_t *data, uint64_t n, uint64_t leaf,
                        uint64_t i, uint8_t out[32])
{
    uint64_t start = i * leaf;
    uint64_t end = start + leaf;
    if (end > n) end = n;
    uint8_t prefix = 0x00;
    osha_ctx c;
    osha_init(&c);
    osha_update(&c, &prefix, 1);
    osha_update(&c, data + start, end - start);
    osha_final(&c, out);
}

/* Interior node: SHA256(0x01 || left || right). */
static void merkle_node(const uint8_t left[32], const uint8_t right[32], uint8_t out[32])
{
    uint8_t msg[65];
    msg[0] = 0x01;
    memcpy(msg + 1, left, 32);
    memcpy(msg + 33, right, 32);
    oracle_sha256(msg, 65, out);
}

uint64_t oracle_merkle_leaf_count(uint64_t n, uint64_t leaf)
{
    if (n == 0 || leaf == 0) return 0;
    return (n + leaf - 1) / leaf;
}

/* Writes every leaf digest (leaf_count * 32 bytes). Returns 0 or -1. */
int oracle_merkle_leaves(const uint8_t *data, uint64_t n, uint64_t leaf, uint8_t *out)
{
    uint64_t nl = oracle_merkle_leaf_count(n, leaf);
    if (nl == 0) return -1;
    for (uint64_t i = 0; i < nl; ++i) merkle_leaf(data, n, leaf, i, out + 32 * i);
    return 0;
}

/* Root of a level of `count` digests, reduced level by level; an unpaired last
 * node is carried up unchanged.  `level` is overwritten.  Returns 0 or -1. */
int oracle_merkle_reduce(uint8_t *level, uint64_t count, uint8_t root[32])
{
    if (count == 0) return -1;
    while (count > 1) {
        uint64_t next = 0;
        for (uint64_t j = 0; j + 1 < count; j += 2) {
            uint8_t parent[32];
            merkle_node(level + 32 * j, level + 32 * (j + 1), parent);
            memcpy(level + 32 * next, parent, 32);
            ++next;
        }
        if (count % 2 == 1) {   /* promotion of the unpaired last node */
            memmove(level + 32 * next, level + 32 * (count - 1), 32);
            ++next;
        }
        count = next;
    }
    memcpy(root, level, 32);
    return 0;
}

/* Root over the n bytes at data with leaves of `leaf` bytes.  Returns 0, or
 * -1 for n == 0, leaf == 0, or an allocation failure. */
int oracle_merkle_root(const uint8_t *data, uint64_t n, uint64_t leaf, uint8_t root[32])
{
    uint64_t nl = oracle_merkle_leaf_count(n, leaf);
    if (nl == 0) return -1;
    uint8_t *level = (uint8_t *)malloc((size_t)(nl * 32));
    if (!level) return -1;
    oracle_merkle_leaves(data, n, leaf, level);
    int rc = oracle_merkle_reduce(level, nl, root);
    free(level);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Whole tree, inclusion proofs, verification                                */
/* [RepOps §2.4: the referee asks for a Merkle membership proof of an input  */
/*  tensor hash against the checkpoint; §2.3.2 checkpoint hash = Merkle tree] */
/* ------------------------------------------------------------------------ */

/* Number of nodes of level l for a tree of nl leaves; levels until one node. */
uint64_t oracle_merkle_total_nodes(uint64_t nl)
{
    if (nl == 0) return 0;
    uint64_t total = 0, count = nl;
    for (;;) {
        total += count;
        if (count == 1) break;
        count = (count + 1) / 2;
    }
    return total;
}

/* Every level, leaf digests first, each level's nodes in index order, 32
 * bytes each; the last node written is the root.  Returns 0 or -1. */
int oracle_merkle_tree(const uint8_t *data, uint64_t n, uint64_t leaf, uint8_t *tree)
{
    uint64_t nl = oracle_merkle_leaf_count(n, leaf);
    if (nl == 0) return -1;
    oracle_merkle_leaves(data, n, leaf, tree);
    uint64_t off = 0, count = nl;
    while (count > 1) {
        uint8_t *cur = tree + 32 * off;
        uint8_t *nxt = cur + 32 * count;
        uint64_t k = 0;
        for (uint64_t j = 0; j + 1 < count; j += 2) merkle_node(cur + 32 * j, cur + 32 * (j + 1), nxt + 32 * k++);
        if (count % 2 == 1) memcpy(nxt + 32 * k++, cur + 32 * (count - 1), 32);
        off += count;
        count = k;
    }
    return 0;
}

/* Siblings of leaf `index`, bottom-up, one per level where the node on the
 * path has a sibling (an unpaired node rises without one).  Writes them to
 * `proof` (32 bytes each) and returns their number, or -1 for a bad index. */
int oracle_merkle_proof(const uint8_t *tree, uint64_t nl, uint64_t index, uint8_t *proof)
{
    if (nl == 0 || index >= nl) return -1;
    uint64_t off = 0, count = nl, j = index;
    int steps = 0;
    while (count > 1) {
        uint64_t sib;
        int has = 1;
        if (j % 2 == 1) sib = j - 1;
        else if (j + 1 < count) sib = j + 1;
        else { has = 0; sib = 0; }
        if (has) memcpy(proof + 32 * steps++, tree + 32 * (off + sib), 32);
        off += count;
        count = (count + 1) / 2;
        j /= 2;
    }
    return steps;
}

/* Recomputes the root from the leaf's bytes, its position and the siblings,
 * and compares it with `root`.  Returns 1 (member), 0 (not), -1 (bad args). */
int oracle_merkle_verify(const uint8_t *leaf_bytes, uint64_t leaf_len, uint64_t nl, uint64_t index,
                         const uint8_t *proof, int steps, const uint8_t root[32])
{
    if (nl == 0 || index >= nl) return -1;
    uint8_t h[32], t[32];
    uint8_t prefix = 0x00;
    osha_ctx c;
    osha_init(&c);
    osha_update(&c, &prefix, 1);
    osha_update(&c, leaf_bytes, leaf_len);
    osha_final(&c, h);
    uint64_t count = nl, j = index;
    int used = 0;
    while (count > 1) {
        if (j % 2 == 1) {
            if (used >= steps) return 0;
            merkle_node(proof + 32 * used++, h, t);
            memcpy(h, t, 32);
        } else if (j + 1 < count) {
            if (used >= steps) return 0;
            merkle_node(h, proof + 32 * used++, t);
            memcpy(h, t, 32);
        }
        count = (count + 1) / 2;
        j /= 2;
    }
    return used == steps && memcmp(h, root, 32) == 0;
}

/* ------------------------------------------------------------------------ */
/* Order-fixed row operators: softmax, LayerNorm, RMSNorm, GeLU              */
/* [RepOps §3.2 (order-critical dimensions run serially or with synchronised */
/*  threads), §3.3 and §4.3 (LayerNorm, GeLU and ERF are the operators that  */
/*  dominate DistilBERT's overhead); §3.1 (the order must not depend on the  */
/*  hardware)]                                                               */
/*                                                                           */
/* The pages fix no algorithm for these operators; the library defines:      */
/*  - reductions over a row in a fixed 32-ary tree: each run of 32           */
/*    consecutive values is folded left to right from its first value; the   */
/*    run results are folded the same way, level by level, until one value   */
/*    is left;                                                               */
/*  - exp by Cody-Waite range reduction x = k*ln2 + r (ln2 split in two      */
/*    parts), a degree-7 Taylor polynomial in r by Horner's rule, and exact  */
/*    scaling by 2^k; every step one rounded IEEE operation, no FMA;         */
/*  - erfc(z), z >= 0, by the Chebyshev fit of Press, Teukolsky, Vetterling  */
/*    and Flannery, Numerical Recipes, section 6.2 (fractional error below   */
/*    1.2e-7), with the exp above;                                           */
/*  - GeLU(x) = 0.5*x*(1 + erf(x/sqrt 2)), with 1 + erf(z) = 2 - erfc(z)     */
/*    for z >= 0 and erfc(-z) for z < 0 (no cancellation);                  */
/*  - a row's normaliser is one correctly rounded reciprocal per row         */
/*    (1/s for softmax, 1/sqrt(var + eps) for the norms), applied to each    */
/*    element by one multiplication.                                         */
/* ------------------------------------------------------------------------ */

#define ROW_RUN 32

/* Fixed 32-ary tree reduction, in place over v[0..n-1]; op 0 = sum, 1 = max.
 * max keeps the earlier value unless the later one is strictly greater. */
static float tree_reduce(float *v, int64_t n, int op)
{
    while (n > 1) {
        int64_t m = 0;
        for (int64_t s = 0; s < n; s += ROW_RUN) {
            int64_t e = s + ROW_RUN < n ? s + ROW_RUN : n;
            float acc = v[s];
            for (int64_t i = s + 1; i < e; ++i) {
                if (op == 0) acc = acc + v[i];
                else if (v[i] > acc) acc = v[i];
            }
            v[m++] = acc;
        }
        n = m;
    }
    return v[0];
}

float oracle_row_sum(const float *x, int64_t n)
{
    float *v = (float *)malloc((size_t)n * sizeof(float));
    memcpy(v, x, (size_t)n * sizeof(float));
    float r = tree_reduce(v, n, 0);
    free(v);
    return r;
}

static float f_from_bits(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }

/* 2^k as a float, for -126 <= k <= 127. */
static float pow2i(int k) { return f_from_bits((uint32_t)(k + 127) << 23); }

float oracle_exp(float x)
{
    if (x != x) return x;
    if (x > 88.72283935546875f) return f_from_bits(0x7f800000u);   /* overflow */
    if (x < -103.972084045410156f) return 0.0f;                    /* below half the least subnormal */
    const float log2e = 1.44269502162933349609375f;   /* float nearest log2(e) */
    const float ln2_hi = 0.693145751953125f;          /* 16 significant bits: k*ln2_hi is exact */
    const float ln2_lo = 1.428606765330187045037746e-06f;
    float t = x * log2e;
    float kf = rintf(t);
    int k = (int)kf;
    float r = x - kf * ln2_hi;
    r = r - kf * ln2_lo;
    /* e^r ~ sum_{i<=7} r^i / i!, Horner from the highest term */
    float p = 1.98412701e-04f;          /* 1/5040 */
    p = p * r + 1.38888892e-03f;        /* 1/720 */
    p = p * r + 8.33333377e-03f;        /* 1/120 */
    p = p * r + 4.16666679e-02f;        /* 1/24 */
    p = p * r + 1.66666672e-01f;        /* 1/6 */
    p = p * r + 0.5f;
    p = p * r + 1.0f;
    p = p * r + 1.0f;
    if (k > 127) return (p * pow2i(127)) * pow2i(k - 127);
    if (k < -126) return (p * pow2i(k + 64)) * pow2i(-64);
    return p * pow2i(k);
}

/* erfc(z) for z >= 0 (Numerical Recipes §6.2 Chebyshev fit). */
float oracle_erfc_pos(float z)
{
    float t = 1.0f / (1.0f + 0.5f * z);
    float q = 0.17087277f;
    q = q * t + -0.82215223f;
    q = q * t + 1.48851587f;
    q = q * t + -1.13520398f;
    q = q * t + 0.27886807f;
    q = q * t + -0.18628806f;
    q = q * t + 0.09678418f;
    q = q * t + 0.37409196f;
    q = q * t + 1.00002368f;
    q = q * t;
    float zz = z * z;
    float arg = (-zz + -1.26551223f) + q;
    return t * oracle_exp(arg);
}

float oracle_gelu(float x)
{
    float z = x * 0.707106769084930419921875f;   /* float nearest 1/sqrt(2) */
    float phi2 = z >= 0.0f ? 2.0f - oracle_erfc_pos(z) : oracle_erfc_pos(-z);
    return (0.5f * x) * phi2;
}

void oracle_gelu_vec(int64_t n, const float *x, float *y)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_gelu(x[i]);
}

/* y_i = e_i * (1/s), e_i = exp(x_i - m), m = tree max of the row, s = tree sum
 * of e, 1/s one correctly rounded division per row. */
void oracle_softmax_rows(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y, int64_t ldy)
{
    float *v = (float *)malloc((size_t)cols * sizeof(float));
    float *e = (float *)malloc((size_t)cols * sizeof(float));
    for (int64_t i = 0; i < rows; ++i) {
        const float *xr = x + i * ldx;
        memcpy(v, xr, (size_t)cols * sizeof(float));
        float m = tree_reduce(v, cols, 1);
        for (int64_t j = 0; j < cols; ++j) e[j] = oracle_exp(xr[j] - m);
        memcpy(v, e, (size_t)cols * sizeof(float));
        float s = tree_reduce(v, cols, 0);
        float inv = 1.0f / s;
        for (int64_t j = 0; j < cols; ++j) y[i * ldy + j] = e[j] * inv;
    }
    free(v);
    free(e);
}

/* Causal softmax: row i is the softmax above over its first
 * L_i = min(cols, first + (i mod period) + 1) values; y[i][j] = +0 for
 * j >= L_i.  (Row i of an attention block whose queries sit at positions
 * first + i sees the keys at positions 0 .. first + i; `period` stacks several
 * heads' blocks of `period` rows.)  first >= 0, period >= 1. */
void oracle_softmax_rows_causal(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y,
                                int64_t ldy, int64_t first, int64_t period)
{
    for (int64_t i = 0; i < rows; ++i) {
        int64_t L = first + i % period + 1;
        if (L > cols) L = cols;
        oracle_softmax_rows(1, L, x + i * ldx, ldx, y + i * ldy, ldy);
        for (int64_t j = L; j < cols; ++j) y[i * ldy + j] = 0.0f;
    }
}

/* mean = sum/n; d = x - mean; var = sum(d*d)/n; inv = 1/sqrt(var + eps);
 * y = (d * inv) * gamma + beta. */
void oracle_layernorm_rows(int64_t rows, int64_t cols, const float *x, int64_t ldx, const float *gamma,
                           const float *beta, float eps, float *y, int64_t ldy)
{
    float *v = (float *)malloc((size_t)cols * sizeof(float));
    float *d = (float *)malloc((size_t)cols * sizeof(float));
    const float n = (float)cols;
    for (int64_t i = 0; i < rows; ++i) {
        const float *xr = x + i * ldx;
        memcpy(v, xr, (size_t)cols * sizeof(float));
        float mean = tree_reduce(v, cols, 0) / n;
        for (int64_t j = 0; j < cols; ++j) { d[j] = xr[j] - mean; v[j] = d[j] * d[j]; }
        float var = tree_reduce(v, cols, 0) / n;
        float inv = 1.0f / sqrtf(var + eps);
        for (int64_t j = 0; j < cols; ++j) y[i * ldy + j] = (d[j] * inv) * gamma[j] + beta[j];
    }
    free(v);
    free(d);
}

/* ms = sum(x*x)/n; inv = 1/sqrt(ms + eps); y = (x * inv) * gamma. */
void oracle_rmsnorm_rows(int64_t rows, int64_t cols, const float *x, int64_t ldx, const float *gamma,
                         float eps, float *y, int64_t ldy)
{
    float *v = (float *)malloc((size_t)cols * sizeof(float));
    const float n = (float)cols;
    for (int64_t i = 0; i < rows; ++i) {
        const float *xr = x + i * ldx;
        for (int64_t j = 0; j < cols; ++j) v[j] = xr[j] * xr[j];
        float ms = tree_reduce(v, cols, 0) / n;
        float inv = 1.0f / sqrtf(ms + eps);
        for (int64_t j = 0; j < cols; ++j) y[i * ldy + j] = (xr[j] * inv) * gamma[j];
    }
    free(v);
}

/* ------------------------------------------------------------------------ */
/* Batched GEMM with a fused epilogue  [RepOps §3.2 matmul example for the   */
/* k-chain; §4.3 (GeLU behind DistilBERT's overhead).  The pages fix no      */
/* epilogue; this is the library's definition.]                             */
/* ------------------------------------------------------------------------ */

/* For b = 0 .. batch-1, with X_b = X + b*strideX for every operand:
 *   acc  = the k-chain of oracle_gemm_f32 for element (i, j) of A_b * B_b;
 *   y    = alpha * acc;
 *   y    = y + bias[j]                  (when bias is not NULL);
 *   y    = GeLU(y)                      (when act == 1);
 *   y    = y + R_b[i*ldr + j]           (when R is not NULL);
 *   C_b[i*ldc + j] = y.
 * Every step is one binary32 rounding.  R may be C itself (same ld and
 * stride): each element reads its residual before it is overwritten.
 *
 * k window (the library's banded reading of a causal product): when
 * k_lo >= 0 the k-chain of row i starts at k = max(0, i - k_lo); when
 * k_hi >= 0 it ends at k = min(K - 1, i + k_hi); -1 leaves that side open.
 * The chain still starts from +0 and runs with k increasing; a row whose
 * window is empty gets the epilogue of +0.
 *
 * b_group >= 1: batch b takes B_(b / b_group) = B + (b / b_group)*strideB
 * (integer division): consecutive batches share one B, as the query heads of
 * a grouped-query attention group share their key/value head. */
void oracle_gemm_batched(int transA, int transB, int64_t batch, int64_t M, int64_t N, int64_t K,
                         const float *A, int64_t lda, int64_t strideA,
                         const float *B, int64_t ldb, int64_t strideB,
                         float *C, int64_t ldc, int64_t strideC,
                         float alpha, const float *bias, int act,
                         const float *R, int64_t ldr, int64_t strideR,
                         int64_t k_lo, int64_t k_hi, int64_t b_group)
{
    for (int64_t b = 0; b < batch; ++b) {
        const float *Ab = A + b * strideA;
        const float *Bb = B + (b / b_group) * strideB;
        float *Cb = C + b * strideC;
        const float *Rb = R ? R + b * strideR : NULL;
        for (int64_t i = 0; i < M; ++i) {
            int64_t k0 = 0, k1 = K;                   /* the chain covers [k0, k1) */
            if (k_lo >= 0 && i - k_lo > k0) k0 = i - k_lo;
            if (k_hi >= 0 && i + k_hi + 1 < k1) k1 = i + k_hi + 1;
            for (int64_t j = 0; j < N; ++j) {
                float acc = 0.0f;
                for (int64_t kk = k0; kk < k1; ++kk) {
                    float a = transA ? Ab[kk * lda + i] : Ab[i * lda + kk];
                    float bv = transB ? Bb[j * ldb + kk] : Bb[kk * ldb + j];
                    float p = a * bv;
                    acc = acc + p;
                }
                float y = alpha * acc;
                if (bias) y = y + bias[j];
                if (act == 1) y = oracle_gelu(y);
                if (Rb) y = y + Rb[i * ldr + j];
                Cb[i * ldc + j] = y;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Half-precision storage  [RepOps §3.3 limitations (IEEE-754 hardware; FP16 */
/* support limited) and §5.3 future work (lower precision such as FP16).     */
/* The pages fix no format rules; the library's: operands stored as IEEE    */
/* binary16 or bfloat16 are widened exactly to binary32, the binary32        */
/* order-fixed path computes, a half output is one round-to-nearest-even.]  */
/* ------------------------------------------------------------------------ */

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float f32_from(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* binary16 -> binary32, exact: subnormals m * 2^-24, normals (1.m) 2^(e-15). */
float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    if (e == 0) {
        float v = (float)m * 5.9604644775390625e-08f;      /* m * 2^-24: exact */
        return f32_from(f32_bits(v) | sign);
    }
    if (e == 31) return f32_from(sign | 0x7f800000u | (m << 13));   /* inf, NaN */
    return f32_from(sign | ((e - 15 + 127) << 23) | (m << 13));
}

/* bfloat16 -> binary32, exact: the 16 bits are the high half. */
float oracle_bf16_to_f32(uint16_t b) { return f32_from((uint32_t)b << 16); }

/* binary32 -> binary16, round to nearest, ties to even.  The value M * 2^E
 * (M the 24-bit significand) is rounded to a multiple of the binary16 quantum
 * 2^Q, Q = max(e - 10, -24) for e = floor(log2 |x|); the count r of quanta
 * gives the encoding ((Q + 24) << 10) + r, which carries into the exponent when
 * r reaches the next power of two.  Past the largest finite value: infinity.
 * NaN: a quiet NaN keeping the top payload bits. */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t x = f32_bits(f);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;
    if (ax > 0x7f800000u) return (uint16_t)(sign | 0x7e00u | ((ax >> 13) & 0x3ffu));
    if (ax == 0x7f800000u) return (uint16_t)(sign | 0x7c00u);
    if (ax == 0) return sign;
    int32_t E;
    uint64_t M;
    if ((ax >> 23) == 0) { M = ax; E = -149; }                       /* binary32 subnormal */
    else { M = (ax & 0x7fffffu) | 0x800000u; E = (int32_t)(ax >> 23) - 127 - 23; }
    int32_t e = E + 23;
    while ((M >> (e - E)) == 0) --e;                                 /* subnormal input: true exponent */
    int32_t Q = e - 10 > -24 ? e - 10 : -24;
    int32_t s = Q - E;                                               /* >= 13 */
    uint64_t r, rem, half;
    if (s > 40) { r = 0; rem = M; half = (uint64_t)1 << 40; }
    else {
        r = M >> s;
        rem = M - (r << s);
        half = (uint64_t)1 << (s - 1);
    }
    if (rem > half || (rem == half && (r & 1))) ++r;
    uint32_t bits = ((uint32_t)(Q + 24) << 10) + (uint32_t)r;
    if (bits >= 0x7c00u) bits = 0x7c00u;
    return (uint16_t)(sign | bits);
}

/* binary32 -> bfloat16, round to nearest, ties to even: bfloat16 keeps the
 * exponent range, so rounding is on the low 16 bits alone -- adding
 * 0x7fff + (bit 16) carries into the kept half exactly when the discarded half
 * is above one half, or equal to it with the kept half odd (a carry out of the
 * largest finite value gives infinity).  NaN: quiet, top payload bits kept. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t x = f32_bits(f);
    if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((x >> 16) | 0x40u);
    uint32_t rounded = x + 0x7fffu + ((x >> 16) & 1u);
    return (uint16_t)(rounded >> 16);
}

static float load_as_f32(const void *p, int64_t i, int type)
{
    if (type == ORACLE_F16) return oracle_f16_to_f32(((const uint16_t *)p)[i]);
    if (type == ORACLE_BF16) return oracle_bf16_to_f32(((const uint16_t *)p)[i]);
    return ((const float *)p)[i];
}

static void store_from_f32(void *p, int64_t i, int type, float v)
{
    if (type == ORACLE_F16) ((uint16_t *)p)[i] = oracle_f32_to_f16(v);
    else if (type == ORACLE_BF16) ((uint16_t *)p)[i] = oracle_f32_to_bf16(v);
    else ((float *)p)[i] = v;
}

/* dst[i] = src[i] converted: widening exact, narrowing round-to-nearest-even. */
void oracle_convert(int64_t n, const void *src, int src_type, void *dst, int dst_type)
{
    for (int64_t i = 0; i < n; ++i) store_from_f32(dst, i, dst_type, load_as_f32(src, i, src_type));
}

/* GEMM on stored operands of any of the three types: every element widened to
 * binary32 (exact), the k-chain of oracle_gemm_f32, the result narrowed once
 * to C's type. */
void oracle_gemm_typed(int64_t M, int64_t N, int64_t K,
                       const void *A, int typeA, int64_t lda, int transA,
                       const void *B, int typeB, int64_t ldb, int transB,
                       void *C, int typeC, int64_t ldc)
{
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            float s = 0.0f;
            for (int64_t q = 0; q < K; ++q) {
                float a = load_as_f32(A, transA ? q * lda + i : i * lda + q, typeA);
                float b = load_as_f32(B, transB ? j * ldb + q : q * ldb + j, typeB);
                float prod = a * b;
                s = s + prod;
            }
            store_from_f32(C, i * ldc + j, typeC, s);
        }
    }
}

/* oracle_mean_sgd with gradients stored as `gtype` (widened exactly); theta
 * stays binary32 (the master weights). */
int oracle_mean_sgd_typed(int nC, int64_t len, const void *const *grads, int gtype,
                          const int *order, float eta, float *theta)
{
    if (nC <= 0) return -1;
    for (int64_t e = 0; e < len; ++e) {
        float S = load_as_f32(grads[order[0]], e, gtype);
        for (int r = 1; r < nC; ++r) S = S + load_as_f32(grads[order[r]], e, gtype);
        float gbar = S / (float)nC;
        float step = eta * gbar;
        float updated = theta[e] - step;
        theta[e] = updated;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Rolling hashes of batch rows  [ZKDV page, proof.start: rolling_window     */
/* hashes within each committed batch row, window at most the row's packed   */
/* width; the protocol commits a rectangular uint32 batch.  The page names   */
/* no hash; the library's: the Rabin-Karp polynomial of the window's words   */
/* modulo the Mersenne prime 2^61 - 1.]                                      */
/* ------------------------------------------------------------------------ */

#define ROLL_P ((((uint64_t)1) << 61) - 1)
#define ROLL_B 4294967311ull     /* the smallest prime above 2^32 */

/* out[r*ldo + i] = (sum_{t<W} words[r*ldw + i + t] * B^(W-1-t)) mod P for every
 * window start i = 0 .. width - W, evaluated directly by Horner's rule. */
void oracle_rolling_hash(int64_t rows, int64_t width, const uint32_t *words, int64_t ldw,
                         int64_t W, uint64_t *out, int64_t ldo)
{
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i + W <= width; ++i) {
            unsigned __int128 h = 0;
            for (int64_t t = 0; t < W; ++t) h = (h * ROLL_B + words[r * ldw + i + t]) % ROLL_P;
            out[r * ldo + i] = (uint64_t)h;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Backward operators of a training step  [RepOps §3.2 (order-critical     */
/* reductions in a fixed order), §4.3 (training: LayerNorm, GeLU, ERF among  */
/* the operators that need reproducible forms).  The pages fix none of      */
/* these; the library's definitions follow, every step one binary32         */
/* rounding, every reduction the 32-ary tree above.]                        */
/* ------------------------------------------------------------------------ */

/* y[j] = tree sum over rows i of x[i*ldx + j]: the column's values in row
 * order, folded by the same 32-ary tree as a row reduction. */
void oracle_colsum(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y)
{
    float *v = (float *)malloc((size_t)(rows > 0 ? rows : 1) * sizeof(float));
    for (int64_t j = 0; j < cols; ++j) {
        for (int64_t i = 0; i < rows; ++i) v[i] = x[i * ldx + j];
        y[j] = rows > 0 ? tree_reduce(v, rows, 0) : 0.0f;
    }
    free(v);
}

/* dx = dy * GeLU'(x), GeLU'(x) = Phi(x) + x * phi(x):
 *   Phi(x) = 0.5 * (1 + erf(x/sqrt 2)), 1 + erf taken as in oracle_gelu;
 *   phi(x) = exp(-(0.5 * x*x)) * (1/sqrt(2 pi)). */
float oracle_gelu_grad(float x)
{
    float z = x * 0.707106769084930419921875f;
    float az = z < 0.0f ? -z : z;
    float e = oracle_erfc_pos(az);
    float phi2 = z >= 0.0f ? 2.0f - e : e;
    float cdf = 0.5f * phi2;
    float xx = x * x;
    float a = -(0.5f * xx);
    float pdf = oracle_exp(a) * 0.3989422917366028f;
    return cdf + x * pdf;
}

void oracle_gelu_backward(int64_t n, const float *x, const float *dy, float *dx)
{
    for (int64_t i = 0; i < n; ++i) dx[i] = dy[i] * oracle_gelu_grad(x[i]);
}

/* RMSNorm backward, per row (forward: inv = 1/sqrt(tree sum(x*x)/n + eps),
 * y = (x * inv) * gamma):
 *   xh = x * inv;  gy = dy * gamma;  c = tree sum(gy * xh) / n;
 *   dx = inv * (gy - xh * c), then + res when res is given (the gradient of a
 *   residual branch around the norm);  dyxh = dy * xh (its column sums are
 *   dgamma).  res may be dx itself. */
void oracle_rmsnorm_backward(int64_t rows, int64_t cols, const float *x, int64_t ldx, const float *gamma,
                             float eps, const float *dy, int64_t lddy, const float *res, int64_t ldres,
                             float *dx, int64_t lddx, float *dyxh, int64_t ldp)
{
    float *v = (float *)malloc((size_t)cols * sizeof(float));
    const float n = (float)cols;
    for (int64_t i = 0; i < rows; ++i) {
        const float *xr = x + i * ldx;
        const float *dr = dy + i * lddy;
        for (int64_t j = 0; j < cols; ++j) v[j] = xr[j] * xr[j];
        float ms = tree_reduce(v, cols, 0) / n;
        float inv = 1.0f / sqrtf(ms + eps);
        for (int64_t j = 0; j < cols; ++j) {
            float xh = xr[j] * inv;
            float gy = dr[j] * gamma[j];
            v[j] = gy * xh;
        }
        float c = tree_reduce(v, cols, 0) / n;
        for (int64_t j = 0; j < cols; ++j) {
            float xh = xr[j] * inv;
            float gy = dr[j] * gamma[j];
            float d = inv * (gy - xh * c);
            if (res) d = d + res[i * ldres + j];
            dx[i * lddx + j] = d;
            dyxh[i * ldp + j] = dr[j] * xh;
        }
    }
    free(v);
}

/* Softmax backward, per row: s = tree sum(dp * p); ds = p * (dp - s).  A
 * causal block's masked entries have p = +0, so their ds is a signed zero. */
void oracle_softmax_backward(int64_t rows, int64_t cols, const float *p, int64_t ldp, const float *dp,
                             int64_t lddp, float *ds, int64_t ldds)
{
    float *v = (float *)malloc((size_t)cols * sizeof(float));
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < cols; ++j) v[j] = dp[i * lddp + j] * p[i * ldp + j];
        float s = tree_reduce(v, cols, 0);
        for (int64_t j = 0; j < cols; ++j) ds[i * ldds + j] = p[i * ldp + j] * (dp[i * lddp + j] - s);
    }
    free(v);
}

/* Causal softmax backward: row i is the backward of the causal softmax's
 * prefix, L_i = min(cols, first + (i mod period) + 1) as in
 * oracle_softmax_rows_causal: s = tree sum over j < L_i of dp_j * p_j (the
 * tree of L_i values), ds_j = p_j * (dp_j - s) for j < L_i and +0 for
 * j >= L_i; nothing beyond the prefix is read. */
void oracle_softmax_backward_causal(int64_t rows, int64_t cols, const float *p, int64_t ldp, const float *dp,
                                    int64_t lddp, float *ds, int64_t ldds, int64_t first, int64_t period)
{
    for (int64_t i = 0; i < rows; ++i) {
        int64_t seen = first + (i % period) + 1;
        if (seen > cols) seen = cols;
        oracle_softmax_backward(1, seen, p + i * ldp, ldp, dp + i * lddp, lddp, ds + i * ldds, ldds);
        for (int64_t j = seen; j < cols; ++j) ds[i * ldds + j] = 0.0f;
    }
}

/* ------------------------------------------------------------------------ */
/* SiLU-gated MLP (SwiGLU) and rotary position embeddings  [RepOps §4.3:    */
/* Llama-style training is the measured workload; the pages fix neither     */
/* operator.  The library's definitions, every step one IEEE rounding.]    */
/* ------------------------------------------------------------------------ */

/* sigma(x) = 1 / (1 + exp(-x)): one correctly rounded division of 1 by
 * (1 + e); exp as oracle_exp (+inf for large -x gives sigma = +0). */
static float sigmoid_fixed(float x)
{
    float e = oracle_exp(-x);
    float den = 1.0f + e;
    return 1.0f / den;
}

/* SiLU(x) = x * sigma(x). */
float oracle_silu(float x)
{
    float sg = sigmoid_fixed(x);
    return x * sg;
}

/* h = SiLU(g) * u, element by element (the gated MLP's hidden activation). */
void oracle_swiglu(int64_t n, const float *g, const float *u, float *h)
{
    for (int64_t i = 0; i < n; ++i) h[i] = oracle_silu(g[i]) * u[i];
}

/* Backward of h = SiLU(g) * u given dh:
 *   du = dh * SiLU(g);
 *   dg = (dh * u) * SiLU'(g),  SiLU'(g) = sigma * (1 + g * (1 - sigma)). */
void oracle_swiglu_backward(int64_t n, const float *g, const float *u, const float *dh, float *dg, float *du)
{
    for (int64_t i = 0; i < n; ++i) {
        float sg = sigmoid_fixed(g[i]);
        float a = g[i] * sg;
        float up = u[i];
        float dhi = dh[i];
        du[i] = dhi * a;
        float t = dhi * up;
        float one_minus = 1.0f - sg;
        float gq = g[i] * one_minus;
        float w = 1.0f + gq;
        float dsilu = sg * w;
        dg[i] = t * dsilu;
    }
}

/* Rotary frequencies: f_i = exp(-((i / pairs) * ln_base)), i = 0 .. pairs-1
 * (base^(-2i/d_head) with pairs = d_head / 2; ln_base is the binary32 value
 * of ln(base) the caller passes).  Each operation one binary32 rounding. */
void oracle_rope_frequencies(int64_t pairs, float ln_base, float *freq)
{
    for (int64_t i = 0; i < pairs; ++i) {
        float frac = (float)i / (float)pairs;
        float x = frac * ln_base;
        freq[i] = oracle_exp(-x);
    }
}

/* cos and sin of a = pos * f, in binary64 with every operation rounded (no
 * FMA), then each rounded once to binary32.  pos * f is exact in binary64
 * (pos < 2^24).  Cody-Waite reduction a = k * (pi/2) + r with pi/2 split in
 * three binary64 parts, the first two of 29 significant bits so that k * part
 * is exact for k < 2^24; Taylor series of sin (to r^15) and cos (to r^16) on
 * |r| <= pi/4 by Horner's rule in z = r^2; the quadrant k mod 4 picks signs
 * and swaps. */
static const double RP_PIO2_1 = 0x1.921fb54p+0;            /* pi/2, leading 29 bits */
static const double RP_PIO2_2 = 0x1.10b4611p-30;           /* next 29 bits */
static const double RP_PIO2_3 = 0x1.4c4c6628b80dcp-59;     /* pi/2 - the two above, rounded */
static const double RP_2_OVER_PI = 0x1.45f306dc9c883p-1;  /* 2/pi, rounded */

static void rope_sincos(int64_t pos, float f, float *c_out, float *s_out)
{
    double a = (double)pos * (double)f;
    double k = rint(a * RP_2_OVER_PI);
    double r = a - k * RP_PIO2_1;
    r = r - k * RP_PIO2_2;
    r = r - k * RP_PIO2_3;
    double z = r * r;
    /* sin r = r + (r z) * q_s;  q_s = -1/3! + z/5! - z^2/7! + ... - z^6/15! */
    double qs = -0x1.ae7f3e733b81fp-41;                   /* -1/15! */
    qs = qs * z + 0x1.6124613a86d09p-33;                 /* 1/13! */
    qs = qs * z + -0x1.ae64567f544e4p-26;                /* -1/11! */
    qs = qs * z + 0x1.71de3a556c734p-19;                 /* 1/9! */
    qs = qs * z + -0x1.a01a01a01a01ap-13;                /* -1/7! */
    qs = qs * z + 0x1.1111111111111p-7;                  /* 1/5! */
    qs = qs * z + -0x1.5555555555555p-3;                 /* -1/3! */
    double rz = r * z;
    double sr = r + rz * qs;
    /* cos r = 1 + z * q_c;  q_c = -1/2! + z/4! - z^2/6! + ... + z^7/16! */
    double qc = 0x1.ae7f3e733b81fp-45;                    /* 1/16! */
    qc = qc * z + -0x1.93974a8c07c9dp-37;                /* -1/14! */
    qc = qc * z + 0x1.1eed8eff8d898p-29;                 /* 1/12! */
    qc = qc * z + -0x1.27e4fb7789f5cp-22;                /* -1/10! */
    qc = qc * z + 0x1.a01a01a01a01ap-16;                 /* 1/8! */
    qc = qc * z + -0x1.6c16c16c16c17p-10;                /* -1/6! */
    qc = qc * z + 0x1.5555555555555p-5;                  /* 1/4! */
    qc = qc * z + -0.5;                                  /* -1/2! */
    double cr = 1.0 + z * qc;
    long long q = (long long)k & 3;
    double sv, cv;
    if (q == 0)      { sv = sr;  cv = cr; }
    else if (q == 1) { sv = cr;  cv = -sr; }
    else if (q == 2) { sv = -sr; cv = -cr; }
    else             { sv = -cr; cv = sr; }
    *c_out = (float)cv;
    *s_out = (float)sv;
}

/* The rotation table: cos[p*pairs + i], sin[p*pairs + i] of angle p * f_i
 * for positions p = 0 .. positions-1. */
void oracle_rope_table(int64_t positions, int64_t pairs, const float *freq, float *cosv, float *sinv)
{
    for (int64_t p = 0; p < positions; ++p)
        for (int64_t i = 0; i < pairs; ++i)
            rope_sincos(p, freq[i], cosv + p * pairs + i, sinv + p * pairs + i);
}

/* Rotates, in place, pair i = (x[2i], x[2i+1]) of every head of every row:
 * row r sits at position pos = first + (r mod period), c = cos[pos][i],
 * s = sin[pos][i];
 *   forward:  (x0 c - x1 s,  x0 s + x1 c)
 *   inverse:  (x0 c + x1 s,  x1 c - x0 s)   (the transpose: the backward).
 * Heads are d_head = 2 * pairs values each, head h at column h * d_head. */
void oracle_rope(int64_t rows, int64_t heads, int64_t pairs, float *x, int64_t ldx, const float *cosv,
                 const float *sinv, int64_t first, int64_t period, int inverse)
{
    for (int64_t r = 0; r < rows; ++r) {
        int64_t pos = first + r % period;
        for (int64_t h = 0; h < heads; ++h) {
            float *v = x + r * ldx + h * 2 * pairs;
            for (int64_t i = 0; i < pairs; ++i) {
                float c = cosv[pos * pairs + i], sn = sinv[pos * pairs + i];
                float x0 = v[2 * i], x1 = v[2 * i + 1];
                float y0, y1;
                if (!inverse) {
                    float a = x0 * c, b = x1 * sn;
                    y0 = a - b;
                    float e = x0 * sn, f = x1 * c;
                    y1 = e + f;
                } else {
                    float a = x0 * c, b = x1 * sn;
                    y0 = a + b;
                    float e = x1 * c, f = x0 * sn;
                    y1 = e - f;
                }
                v[2 * i] = y0;
                v[2 * i + 1] = y1;
            }
        }
    }
}
