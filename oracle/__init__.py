"""CPU oracle for the reproducible-operator hot path -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg may
import this package.  The product path (the CUDA library and its Python
binding) never does, and fails loudly when its own extension is missing.

The arithmetic lives in `repops_oracle.c` (plain single-threaded C, built with
-ffp-contract=off).  This module only marshals numpy arrays through ctypes.

What each function follows (page title, section):
  gemm       -- "Verde与RepOps" §3.2, the matmul example: any order over i, j;
                k strictly increasing from sum = 0; sum = sum + a*b with the
                product and the sum each rounded to binary32 (no FMA, as
                "Zoo Per-LLM Chain Soundness" §5 "Determinism of left-fold" pins).
  sort_ids   -- "Zoo Per-LLM Chain Soundness" §2 Lemma "Order independence
                within a batch" and §5 "Ordering subroutine": contributors in
                lexicographic DID byte order.
  mean_sgd   -- same page, §2 Definition "Aggregation rule" (mean over the
                contributor set), §5 "Ordering subroutine" (left fold in sorted
                order, scaled by 1/k) and "Update step" (theta -= eta * gbar).
  sha256     -- FIPS 180-4 (the pages name no hash; SHA-256 is the reading taken).
  merkle_*   -- "Zoo Per-LLM Chain Soundness" §1 (batch hash = Merkle root),
                §6 (bytes32 roots); "Verde与RepOps" §2.3.2 (checkpoint hash is a
                Merkle tree) and §2.4 (membership proofs).
  exp, erfc_pos, gelu, row_sum, softmax_rows, layernorm_rows, rmsnorm_rows
             -- "Verde与RepOps" §3.2 (order-critical dimensions serial or with
                synchronised threads), §4.3 (LayerNorm, GeLU, ERF): reductions in
                a fixed 32-ary tree, exp by Cody-Waite reduction + Horner, erfc
                by the Numerical Recipes §6.2 Chebyshev fit (see the C source).
  silu, swiglu, swiglu_backward, rope_frequencies, rope_table, rope,
  softmax_backward_causal, gemm_batched(k_lo, k_hi)
             -- "Verde与RepOps" §4.3 (Llama-style training as the workload); the
                pages fix none of these; the library's definitions are in the
                C source, each step one IEEE rounding.
  replay     -- "Zoo Per-LLM Chain Soundness" §7 "Reproducibility test plan":
                replay each block's batch in order, then check H(theta) = m.
Pins against things other than the oracle itself live in tests/test_oracle_*.py.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    """Loads (building first if needed) the oracle shared library.

    REPOPS_ORACLE_LIB names another build of repops_oracle.c to load instead;
    the mutation tests use it to show that the pins catch planted mistakes."""
    global _lib
    if _lib is None:
        path = os.environ.get("REPOPS_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.oracle_fp_env_ok.restype = i32
        L.oracle_fp_env_ok.argtypes = []
        L.oracle_gemm_f32.restype = None
        L.oracle_gemm_f32.argtypes = [i64, i64, i64, vp, i64, i32, vp, i64, i32, vp, i64]
        L.oracle_sort_ids.restype = i32
        L.oracle_sort_ids.argtypes = [i32, vp, vp, vp, vp]
        L.oracle_mean_sgd.restype = i32
        L.oracle_mean_sgd.argtypes = [i32, i64, vp, vp, ctypes.c_float, vp]
        L.oracle_sha256.restype = None
        L.oracle_sha256.argtypes = [vp, ctypes.c_uint64, vp]
        L.oracle_sha256_constants.restype = None
        L.oracle_sha256_constants.argtypes = [vp, vp]
        L.oracle_merkle_leaf_count.restype = ctypes.c_uint64
        L.oracle_merkle_leaf_count.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.oracle_merkle_leaves.restype = i32
        L.oracle_merkle_leaves.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint64, vp]
        L.oracle_merkle_reduce.restype = i32
        L.oracle_merkle_reduce.argtypes = [vp, ctypes.c_uint64, vp]
        L.oracle_merkle_root.restype = i32
        L.oracle_merkle_root.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint64, vp]
        L.oracle_merkle_total_nodes.restype = ctypes.c_uint64
        L.oracle_merkle_total_nodes.argtypes = [ctypes.c_uint64]
        L.oracle_merkle_tree.restype = i32
        L.oracle_merkle_tree.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint64, vp]
        L.oracle_merkle_proof.restype = i32
        L.oracle_merkle_proof.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint64, vp]
        L.oracle_merkle_verify.restype = i32
        L.oracle_merkle_verify.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, vp,
                                           i32, vp]
        f32 = ctypes.c_float
        L.oracle_exp.restype = f32
        L.oracle_exp.argtypes = [f32]
        L.oracle_erfc_pos.restype = f32
        L.oracle_erfc_pos.argtypes = [f32]
        L.oracle_gelu.restype = f32
        L.oracle_gelu.argtypes = [f32]
        L.oracle_gelu_vec.restype = None
        L.oracle_gelu_vec.argtypes = [i64, vp, vp]
        L.oracle_row_sum.restype = f32
        L.oracle_row_sum.argtypes = [vp, i64]
        L.oracle_softmax_rows.restype = None
        L.oracle_softmax_rows.argtypes = [i64, i64, vp, i64, vp, i64]
        L.oracle_layernorm_rows.restype = None
        L.oracle_layernorm_rows.argtypes = [i64, i64, vp, i64, vp, vp, f32, vp, i64]
        L.oracle_rmsnorm_rows.restype = None
        L.oracle_rmsnorm_rows.argtypes = [i64, i64, vp, i64, vp, f32, vp, i64]
        L.oracle_softmax_rows_causal.restype = None
        L.oracle_softmax_rows_causal.argtypes = [i64, i64, vp, i64, vp, i64, i64, i64]
        L.oracle_convert.restype = None
        L.oracle_convert.argtypes = [i64, vp, i32, vp, i32]
        L.oracle_gemm_typed.restype = None
        L.oracle_gemm_typed.argtypes = [i64, i64, i64, vp, i32, i64, i32, vp, i32, i64, i32, vp, i32, i64]
        L.oracle_mean_sgd_typed.restype = i32
        L.oracle_mean_sgd_typed.argtypes = [i32, i64, vp, i32, vp, f32, vp]
        L.oracle_rolling_hash.restype = None
        L.oracle_rolling_hash.argtypes = [i64, i64, vp, i64, i64, vp, i64]
        L.oracle_colsum.restype = None
        L.oracle_colsum.argtypes = [i64, i64, vp, i64, vp]
        L.oracle_gelu_grad.restype = f32
        L.oracle_gelu_grad.argtypes = [f32]
        L.oracle_gelu_backward.restype = None
        L.oracle_gelu_backward.argtypes = [i64, vp, vp, vp]
        L.oracle_rmsnorm_backward.restype = None
        L.oracle_rmsnorm_backward.argtypes = [i64, i64, vp, i64, vp, f32, vp, i64, vp, i64, vp, i64, vp, i64]
        L.oracle_softmax_backward.restype = None
        L.oracle_softmax_backward.argtypes = [i64, i64, vp, i64, vp, i64, vp, i64]
        L.oracle_gemm_batched.restype = None
        L.oracle_gemm_batched.argtypes = [i32, i32, i64, i64, i64, i64, vp, i64, i64, vp, i64, i64,
                                          vp, i64, i64, f32, vp, i32, vp, i64, i64, i64, i64, i64]
        L.oracle_softmax_backward_causal.restype = None
        L.oracle_softmax_backward_causal.argtypes = [i64, i64, vp, i64, vp, i64, vp, i64, i64, i64]
        L.oracle_silu.restype = f32
        L.oracle_silu.argtypes = [f32]
        L.oracle_swiglu.restype = None
        L.oracle_swiglu.argtypes = [i64, vp, vp, vp]
        L.oracle_swiglu_backward.restype = None
        L.oracle_swiglu_backward.argtypes = [i64, vp, vp, vp, vp, vp]
        L.oracle_rope_frequencies.restype = None
        L.oracle_rope_frequencies.argtypes = [i64, f32, vp]
        L.oracle_rope_table.restype = None
        L.oracle_rope_table.argtypes = [i64, i64, vp, vp, vp]
        L.oracle_rope.restype = None
        L.oracle_rope.argtypes = [i64, i64, i64, vp, i64, vp, vp, i64, i64, i32]
        if L.oracle_fp_env_ok() != 1:
            raise RuntimeError("host floating-point environment flushes subnormals "
                               "or does not round to nearest even; the oracle "
                               "would not be the IEEE-754 binary32 reference")
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _operand(X: np.ndarray):
    """(base array, leading dim, transposed flag) for a 2-D float32 view."""
    if X.dtype != np.float32 or X.ndim != 2:
        raise TypeError("expected a 2-D float32 array")
    r, c = X.shape
    s0, s1 = (s // 4 for s in X.strides)
    if X.strides[0] % 4 or X.strides[1] % 4:
        X = np.ascontiguousarray(X)
        s0, s1 = c, 1
    if s1 == 1 and s0 >= max(c, 1):
        return X, s0, 0
    if s0 == 1 and s1 >= max(r, 1):
        return X, s1, 1
    X = np.ascontiguousarray(X)
    return X, max(c, 1), 0


def gemm(A: np.ndarray, B: np.ndarray, out: np.ndarray = None) -> np.ndarray:
    """C = A @ B with the order-fixed, separately rounded k-chain.

    A (M x K) and B (K x N) may be row-major or transposed (column-major)
    views; the element values are what count, not the storage."""
    L = lib()
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    A_, lda, ta = _operand(A)
    B_, ldb, tb = _operand(B)
    C = out if out is not None else np.empty((M, N), dtype=np.float32)
    if C.dtype != np.float32 or C.strides[1] != 4:
        raise TypeError("out must be float32 with unit column stride")
    if M and N:
        L.oracle_gemm_f32(M, N, K, _ptr(A_), lda, ta, _ptr(B_), ldb, tb,
                          _ptr(C), C.strides[0] // 4)
    return C


def sort_ids(ids) -> list:
    """Indices of `ids` (a sequence of bytes) in lexicographic unsigned byte order."""
    L = lib()
    n = len(ids)
    blob = b"".join(ids)
    buf = np.frombuffer(blob, dtype=np.uint8).copy() if blob else np.zeros(1, np.uint8)
    lens = np.array([len(x) for x in ids], dtype=np.int64)
    offs = np.zeros(n, dtype=np.int64)
    if n > 1:
        offs[1:] = np.cumsum(lens)[:-1]
    order = np.zeros(max(n, 1), dtype=np.int32)
    rc = L.oracle_sort_ids(n, _ptr(buf), _ptr(offs), _ptr(lens), _ptr(order))
    if rc != 0:
        raise ValueError("duplicate contributor identifiers")
    return [int(x) for x in order[:n]]


def mean_sgd(grads, order, eta: float, theta: np.ndarray) -> np.ndarray:
    """Returns a new theta: theta - eta * (left fold of grads in `order`) / |C|."""
    L = lib()
    nC = len(grads)
    th = np.array(theta, dtype=np.float32, copy=True)
    gs = [np.ascontiguousarray(g, dtype=np.float32) for g in grads]
    for g in gs:
        if g.shape != th.shape:
            raise ValueError("gradient and theta shapes differ")
    ptrs = (ctypes.c_void_p * max(nC, 1))(*[_ptr(g) for g in gs])
    o = np.array(list(order), dtype=np.int32)
    if o.size != nC:
        raise ValueError("order must have one entry per contributor")
    rc = L.oracle_mean_sgd(nC, th.size, ctypes.cast(ptrs, ctypes.c_void_p),
                           _ptr(o) if nC else None, ctypes.c_float(eta), _ptr(th))
    if rc != 0:
        raise ValueError("order is not a permutation of the contributors")
    return th


def _as_bytes(data) -> np.ndarray:
    if isinstance(data, (bytes, bytearray, memoryview)):
        return np.frombuffer(bytes(data), dtype=np.uint8)
    a = np.ascontiguousarray(data)
    return a.reshape(-1).view(np.uint8)


def sha256(data) -> bytes:
    L = lib()
    b = _as_bytes(data)
    out = np.zeros(32, dtype=np.uint8)
    L.oracle_sha256(_ptr(b) if b.size else None, b.size, _ptr(out))
    return out.tobytes()


def sha256_constants():
    """(K[64], H0[8]) derived from the primes, FIPS 180-4 §4.2.2 and §5.3.3."""
    L = lib()
    K = np.zeros(64, dtype=np.uint32)
    H = np.zeros(8, dtype=np.uint32)
    L.oracle_sha256_constants(_ptr(K), _ptr(H))
    return [int(x) for x in K], [int(x) for x in H]


def merkle_leaves(data, leaf: int = 4096) -> np.ndarray:
    """(leaf_count, 32) uint8 array of leaf digests SHA256(0x00 || leaf bytes)."""
    L = lib()
    b = _as_bytes(data)
    n = L.oracle_merkle_leaf_count(b.size, leaf)
    if n == 0:
        raise ValueError("empty input or zero leaf size")
    out = np.zeros((n, 32), dtype=np.uint8)
    L.oracle_merkle_leaves(_ptr(b), b.size, leaf, _ptr(out))
    return out


def merkle_reduce(digests: np.ndarray) -> bytes:
    """Root over a level of 32-byte digests (pairs hashed with 0x01, odd promoted)."""
    L = lib()
    lv = np.array(digests, dtype=np.uint8, copy=True).reshape(-1, 32)
    if lv.shape[0] == 0:
        raise ValueError("empty level")
    root = np.zeros(32, dtype=np.uint8)
    L.oracle_merkle_reduce(_ptr(lv), lv.shape[0], _ptr(root))
    return root.tobytes()


def merkle_root(data, leaf: int = 4096) -> bytes:
    """32-byte Merkle root over the bytes of `data` with `leaf`-byte leaves."""
    L = lib()
    b = _as_bytes(data)
    root = np.zeros(32, dtype=np.uint8)
    rc = L.oracle_merkle_root(_ptr(b) if b.size else None, b.size, leaf, _ptr(root))
    if rc != 0:
        raise ValueError("empty input or zero leaf size")
    return root.tobytes()


def merkle_tree(data, leaf: int = 4096) -> np.ndarray:
    """(total_nodes, 32) uint8: every level, leaf digests first; last row = root."""
    L = lib()
    b = _as_bytes(data)
    nl = L.oracle_merkle_leaf_count(b.size, leaf)
    if nl == 0:
        raise ValueError("empty input or zero leaf size")
    out = np.zeros((L.oracle_merkle_total_nodes(nl), 32), dtype=np.uint8)
    L.oracle_merkle_tree(_ptr(b), b.size, leaf, _ptr(out))
    return out


def merkle_proof(tree: np.ndarray, nleaves: int, index: int) -> np.ndarray:
    """(steps, 32) uint8 siblings of leaf `index`, bottom-up."""
    L = lib()
    t = np.ascontiguousarray(tree, dtype=np.uint8)
    buf = np.zeros((64, 32), dtype=np.uint8)
    n = L.oracle_merkle_proof(_ptr(t), nleaves, index, _ptr(buf))
    if n < 0:
        raise ValueError("leaf index out of range")
    return buf[:n].copy()


def merkle_verify(leaf_bytes, nleaves: int, index: int, proof, root: bytes) -> bool:
    """Membership of a leaf's bytes at `index` in the tree with this root."""
    L = lib()
    lb = _as_bytes(leaf_bytes)
    pf = np.ascontiguousarray(np.asarray(proof, dtype=np.uint8).reshape(-1, 32))
    r = np.frombuffer(bytes(root), dtype=np.uint8).copy()
    rc = L.oracle_merkle_verify(_ptr(lb) if lb.size else None, lb.size, nleaves, index,
                                _ptr(pf) if pf.size else None, pf.shape[0], _ptr(r))
    if rc < 0:
        raise ValueError("leaf index out of range")
    return rc == 1


def replay(grads_per_step, orders, etas, theta, leaf: int = 4096):
    """theta_t = mean_sgd(theta_{t-1}, G_t) and m_t = root(theta_t) per step.

    Returns (final theta, [m_1, ..., m_T])."""
    th = np.array(theta, dtype=np.float32, copy=True)
    roots = []
    for gs, order, eta in zip(grads_per_step, orders, etas):
        th = mean_sgd(gs, order, eta, th)
        roots.append(merkle_root(th, leaf))
    return th, roots


def exp(x: float) -> float:
    return float(lib().oracle_exp(ctypes.c_float(x)))


def erfc_pos(z: float) -> float:
    return float(lib().oracle_erfc_pos(ctypes.c_float(z)))


def gelu(x) -> np.ndarray:
    L = lib()
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(a)
    L.oracle_gelu_vec(a.size, _ptr(a), _ptr(out))
    return out


def row_sum(x) -> float:
    a = np.ascontiguousarray(x, dtype=np.float32)
    return float(lib().oracle_row_sum(_ptr(a), a.size))


def _rows(x):
    a = np.asarray(x, dtype=np.float32)
    if a.ndim != 2 or a.strides[1] != 4:
        a = np.ascontiguousarray(a)
    return a, a.strides[0] // 4


def softmax_rows(x) -> np.ndarray:
    a, lda = _rows(x)
    y = np.empty(a.shape, dtype=np.float32)
    lib().oracle_softmax_rows(a.shape[0], a.shape[1], _ptr(a), lda, _ptr(y), a.shape[1])
    return y


def layernorm_rows(x, gamma, beta, eps: float) -> np.ndarray:
    a, lda = _rows(x)
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    b = np.ascontiguousarray(beta, dtype=np.float32)
    y = np.empty(a.shape, dtype=np.float32)
    lib().oracle_layernorm_rows(a.shape[0], a.shape[1], _ptr(a), lda, _ptr(g), _ptr(b),
                                ctypes.c_float(eps), _ptr(y), a.shape[1])
    return y


def rmsnorm_rows(x, gamma, eps: float) -> np.ndarray:
    a, lda = _rows(x)
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    y = np.empty(a.shape, dtype=np.float32)
    lib().oracle_rmsnorm_rows(a.shape[0], a.shape[1], _ptr(a), lda, _ptr(g), ctypes.c_float(eps),
                              _ptr(y), a.shape[1])
    return y


ACT_NONE, ACT_GELU = 0, 1


def gemm_batched(transA, transB, batch, M, N, K, A, lda, strideA, B, ldb, strideB,
                 C, ldc, strideC, alpha=1.0, bias=None, act=ACT_NONE, R=None, ldr=0, strideR=0,
                 k_lo=-1, k_hi=-1, b_group=1):
    """Batched GEMM with the fused epilogue, on flat float32 buffers (element
    offsets and strides exactly as the library's batched entry point takes
    them).  C is written in place; R may be C itself.  k_lo / k_hi >= 0
    restrict row i's k-chain to [i - k_lo, i + k_hi]; b_group > 1 lets
    b_group consecutive batches share one B (see the C source)."""
    L = lib()
    for X in (A, B, C) + tuple(x for x in (bias, R) if x is not None):
        if X.dtype != np.float32 or not X.flags.c_contiguous:
            raise TypeError("flat contiguous float32 buffers expected")
    L.oracle_gemm_batched(int(bool(transA)), int(bool(transB)), batch, M, N, K,
                          _ptr(A), lda, strideA, _ptr(B), ldb, strideB, _ptr(C), ldc, strideC,
                          float(alpha), _ptr(bias) if bias is not None else None, int(act),
                          _ptr(R) if R is not None else None, ldr, strideR, int(k_lo), int(k_hi), int(b_group))
    return C


def softmax_rows_causal(X: np.ndarray, first: int, period: int = None) -> np.ndarray:
    """Row i: softmax over its first min(cols, first + (i mod period) + 1)
    values, +0 after (period defaults to the row count: no repetition)."""
    L = lib()
    X = np.ascontiguousarray(X, dtype=np.float32)
    rows, cols = X.shape
    Y = np.empty_like(X)
    if rows and cols:
        L.oracle_softmax_rows_causal(rows, cols, _ptr(X), cols, _ptr(Y), cols, first, period or rows)
    return Y


F32, F16, BF16 = 0, 1, 2


def _storage(a, t):
    """Flat contiguous buffer of storage type t (F32: float32; F16/BF16: uint16 bits)."""
    return np.ascontiguousarray(a, dtype=np.float32 if t == F32 else np.uint16)


def convert(x, src_type: int, dst_type: int) -> np.ndarray:
    """Element-wise conversion between stored types (exact widening, round to
    nearest even narrowing); half types travel as their uint16 bit patterns."""
    a = _storage(x, src_type)
    out = np.empty(a.shape, dtype=np.float32 if dst_type == F32 else np.uint16)
    if a.size:
        lib().oracle_convert(a.size, _ptr(a), src_type, _ptr(out), dst_type)
    return out


def gemm_typed(A, typeA: int, B, typeB: int, typeC: int) -> np.ndarray:
    """C = A @ B on stored operands (row-major 2-D arrays of their storage
    type), computed on the exactly widened values, narrowed once to typeC."""
    L = lib()
    A_ = _storage(A, typeA)
    B_ = _storage(B, typeB)
    M, K = A_.shape
    N = B_.shape[1]
    C = np.empty((M, N), dtype=np.float32 if typeC == F32 else np.uint16)
    if M and N:
        L.oracle_gemm_typed(M, N, K, _ptr(A_), typeA, max(K, 1), 0, _ptr(B_), typeB, max(N, 1), 0,
                            _ptr(C), typeC, max(N, 1))
    return C


def mean_sgd_typed(grads, gtype: int, order, eta: float, theta: np.ndarray) -> np.ndarray:
    """As mean_sgd with gradients stored as gtype; returns a new float32 theta."""
    L = lib()
    th = np.array(theta, dtype=np.float32, copy=True)
    gs = [_storage(g, gtype) for g in grads]
    ptrs = (ctypes.c_void_p * max(len(gs), 1))(*[_ptr(g) for g in gs])
    o = np.ascontiguousarray(order, dtype=np.int32)
    rc = L.oracle_mean_sgd_typed(len(gs), th.size, ctypes.cast(ptrs, ctypes.c_void_p), gtype, _ptr(o),
                                 ctypes.c_float(eta), _ptr(th))
    if rc != 0:
        raise ValueError("bad contributor set")
    return th


def rolling_hash(words: np.ndarray, window: int) -> np.ndarray:
    """(rows, width - window + 1) uint64 window hashes of a (rows, width) uint32 batch."""
    w = np.ascontiguousarray(words, dtype=np.uint32)
    rows, width = w.shape
    n = width - window + 1
    out = np.empty((rows, max(n, 0)), dtype=np.uint64)
    if rows and n > 0:
        lib().oracle_rolling_hash(rows, width, _ptr(w), width, window, _ptr(out), n)
    return out


def colsum(x) -> np.ndarray:
    """Column sums of a 2-D float32 array, each over the 32-ary tree in row order."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(a.shape[1], dtype=np.float32)
    if a.shape[1]:
        lib().oracle_colsum(a.shape[0], a.shape[1], _ptr(a), a.shape[1], _ptr(y))
    return y


def gelu_grad(x: float) -> float:
    return lib().oracle_gelu_grad(float(x))


def gelu_backward(x, dy) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32)
    d = np.ascontiguousarray(dy, dtype=np.float32)
    out = np.empty_like(a)
    lib().oracle_gelu_backward(a.size, _ptr(a), _ptr(d), _ptr(out))
    return out


def rmsnorm_backward(x, gamma, eps: float, dy, res=None):
    """(dx, dy * xhat) of RMSNorm rows, dx + res when res is given;
    dgamma = colsum(dy * xhat)."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    d = np.ascontiguousarray(dy, dtype=np.float32)
    rr = np.ascontiguousarray(res, dtype=np.float32) if res is not None else None
    dx = np.empty_like(a)
    pr = np.empty_like(a)
    r, c = a.shape
    lib().oracle_rmsnorm_backward(r, c, _ptr(a), c, _ptr(g), ctypes.c_float(eps), _ptr(d), c,
                                  _ptr(rr) if rr is not None else None, c, _ptr(dx), c, _ptr(pr), c)
    return dx, pr


def softmax_backward(p, dp) -> np.ndarray:
    a = np.ascontiguousarray(p, dtype=np.float32)
    d = np.ascontiguousarray(dp, dtype=np.float32)
    out = np.empty_like(a)
    r, c = a.shape
    lib().oracle_softmax_backward(r, c, _ptr(a), c, _ptr(d), c, _ptr(out), c)
    return out


def softmax_backward_causal(p, dp, first: int, period: int = None) -> np.ndarray:
    """Row i: the softmax backward over its first min(cols, first + (i mod
    period) + 1) entries, +0 after (period defaults to the row count)."""
    a = np.ascontiguousarray(p, dtype=np.float32)
    d = np.ascontiguousarray(dp, dtype=np.float32)
    out = np.empty_like(a)
    r, c = a.shape
    if r and c:
        lib().oracle_softmax_backward_causal(r, c, _ptr(a), c, _ptr(d), c, _ptr(out), c, first, period or r)
    return out


def silu(x: float) -> float:
    return float(lib().oracle_silu(ctypes.c_float(x)))


def swiglu(g, u) -> np.ndarray:
    """SiLU(g) * u element by element."""
    a = np.ascontiguousarray(g, dtype=np.float32)
    b = np.ascontiguousarray(u, dtype=np.float32)
    out = np.empty_like(a)
    lib().oracle_swiglu(a.size, _ptr(a), _ptr(b), _ptr(out))
    return out


def swiglu_backward(g, u, dh):
    """(dg, du) of h = SiLU(g) * u given dh."""
    a = np.ascontiguousarray(g, dtype=np.float32)
    b = np.ascontiguousarray(u, dtype=np.float32)
    d = np.ascontiguousarray(dh, dtype=np.float32)
    dg, du = np.empty_like(a), np.empty_like(a)
    lib().oracle_swiglu_backward(a.size, _ptr(a), _ptr(b), _ptr(d), _ptr(dg), _ptr(du))
    return dg, du


def rope_frequencies(pairs: int, ln_base: float) -> np.ndarray:
    out = np.empty(pairs, np.float32)
    lib().oracle_rope_frequencies(pairs, ctypes.c_float(ln_base), _ptr(out))
    return out


def rope_table(positions: int, freq):
    """(cos, sin), each positions x pairs, of angle p * freq[i]."""
    f = np.ascontiguousarray(freq, dtype=np.float32)
    c = np.empty((positions, f.size), np.float32)
    s = np.empty((positions, f.size), np.float32)
    lib().oracle_rope_table(positions, f.size, _ptr(f), _ptr(c), _ptr(s))
    return c, s


def rope(x, heads: int, cos, sin, first: int = 0, period: int = None, inverse: bool = False) -> np.ndarray:
    """Returns x (rows x heads*d_head, at least) with every head's pairs
    rotated to row r's position first + (r mod period)."""
    a = np.array(x, dtype=np.float32, order="C", copy=True)
    c = np.ascontiguousarray(cos, dtype=np.float32)
    s = np.ascontiguousarray(sin, dtype=np.float32)
    rows, cols = a.shape
    if rows:
        lib().oracle_rope(rows, heads, c.shape[1], _ptr(a), cols, _ptr(c), _ptr(s), first, period or rows,
                          int(bool(inverse)))
    return a
