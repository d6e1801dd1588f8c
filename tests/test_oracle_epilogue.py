"""Pins the oracle's batched GEMM with the fused epilogue.

Sources: "Verde与RepOps" §3.2 (the k-chain: k strictly increasing from +0, every
product and sum rounded on its own); §4.3 (GeLU among the operators behind
DistilBERT's overhead).  The pages fix no epilogue; the library's definition --
y = alpha*acc, then + bias[j], then GeLU, then + residual, each one binary32
rounding -- is restated here in exact rational arithmetic with independent
indexing code, on every storage option, stride pattern and epilogue part.
"""
import itertools

import numpy as np
import pytest

import fp32_exact as fx


def elem(buf, off):
    return float(buf[off])


def ref_batched(orc, transA, transB, batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC,
                alpha, bias, act, R, ldr, sR, group=1):
    """Element-by-element restatement; returns the new contents of C.  Batch
    b reads the B of batch b // group."""
    out = C.copy()
    old = C.copy()                       # an in-place residual reads the old C
    src_R = old if R is C else R
    for b in range(batch):
        for i in range(M):
            for j in range(N):
                s = 0.0
                for k in range(K):
                    a = elem(A, b * sA + (k * lda + i if transA else i * lda + k))
                    w = elem(B, (b // group) * sB + (j * ldb + k if transB else k * ldb + j))
                    s = fx.add(s, fx.mul(a, w))
                y = fx.mul(s, float(np.float32(alpha)))
                if bias is not None:
                    y = fx.add(y, float(bias[j]))
                if act == 1:
                    y = float(orc.gelu(np.array([y], np.float32))[0])
                if R is not None:
                    y = fx.add(y, elem(src_R, b * sR + i * ldr + j))
                out[b * sC + i * ldc + j] = y
    return out


def wide(rng, n):
    v = (rng.uniform(-1, 1, n) * np.exp2(rng.integers(-12, 12, n))).astype(np.float32)
    v[rng.random(n) < 0.05] = 0.0
    return v


def layout(kind, batch, rows, cols, pad):
    """(ld, stride, buffer length) of `batch` rows x cols matrices."""
    if kind == "stacked":
        ld = cols + pad
        stride = rows * ld + pad
    elif kind == "interleaved":             # matrix b occupies columns [b*cols, (b+1)*cols)
        ld = batch * cols + pad
        stride = cols
    else:                                   # "broadcast": every batch reads matrix 0
        ld = cols + pad
        stride = 0
    return ld, stride, (batch - 1) * stride + (rows - 1) * ld + cols + 3


CASES = list(itertools.product([0, 1], [0, 1], ["stacked", "interleaved", "broadcast"]))


@pytest.mark.parametrize("transA,transB,kind", CASES)
def test_batched_epilogue_exact_rational(orc, transA, transB, kind):
    rng = np.random.default_rng(17 + 4 * transA + 2 * transB + len(kind))
    batch, M, N, K = 3, 4, 5, 6
    ar, ac = (K, M) if transA else (M, K)
    br, bc = (N, K) if transB else (K, N)
    lda, sA, la = layout(kind, batch, ar, ac, 1)
    ldb, sB, lb = layout("stacked" if kind == "broadcast" else kind, batch, br, bc, 2)
    ldc, sC, lc = layout("interleaved" if kind == "interleaved" else "stacked", batch, M, N, 1)
    A, B = wide(rng, la), wide(rng, lb)
    bias = wide(rng, N)
    R = wide(rng, lc)
    for alpha, with_bias, act, with_R in [(1.0, False, 0, False), (3.0, True, 0, False),
                                          (0.125, False, 1, False), (-1.5, True, 1, True),
                                          (1.0, False, 0, True)]:
        C = wide(rng, lc)
        want = ref_batched(orc, transA, transB, batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC,
                           alpha, bias if with_bias else None, act, R if with_R else None, ldc, sC)
        orc.gemm_batched(transA, transB, batch, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, alpha,
                         bias if with_bias else None, act, R if with_R else None, ldc, sC)
        assert [fx.bits(float(v)) for v in C] == [fx.bits(float(v)) for v in want]


@pytest.mark.parametrize("group,transB", [(2, 0), (3, 1), (6, 0)])
def test_grouped_b_exact_rational(orc, group, transB):
    # six batches whose B is shared by `group` consecutive ones (grouped-query
    # attention: the query heads of a group share one key/value head)
    rng = np.random.default_rng(40 + group + transB)
    batch, M, N, K = 6, 3, 4, 5
    br, bc = (N, K) if transB else (K, N)
    nb = -(-batch // group)
    A, B = wide(rng, batch * M * K), wide(rng, nb * br * bc)
    C = np.zeros(batch * M * N, np.float32)
    want = ref_batched(orc, 0, transB, batch, M, N, K, A, K, M * K, B, bc, br * bc, C, N, M * N,
                       0.5, None, 0, None, N, M * N, group=group)
    orc.gemm_batched(0, transB, batch, M, N, K, A, K, M * K, B, bc, br * bc, C, N, M * N, 0.5, b_group=group)
    assert [fx.bits(float(v)) for v in C] == [fx.bits(float(v)) for v in want]


def test_in_place_residual(orc):
    rng = np.random.default_rng(5)
    batch, M, N, K = 2, 3, 4, 5
    A = wide(rng, batch * M * K)
    B = wide(rng, batch * K * N)
    C = wide(rng, batch * M * N)
    bias = wide(rng, N)
    want = ref_batched(orc, 0, 0, batch, M, N, K, A, K, M * K, B, N, K * N, C, N, M * N,
                       2.0, bias, 1, C, N, M * N)
    orc.gemm_batched(0, 0, batch, M, N, K, A, K, M * K, B, N, K * N, C, N, M * N, 2.0, bias, 1, C, N, M * N)
    assert [fx.bits(float(v)) for v in C] == [fx.bits(float(v)) for v in want]


def test_integer_closed_form(orc):
    # small integers: every product, sum and epilogue step is exact, so
    # C_b = alpha * A_b B + bias + R_b in exact arithmetic (B broadcast)
    rng = np.random.default_rng(9)
    batch, M, N, K = 4, 7, 9, 33
    A = rng.integers(-8, 9, (batch, M, K)).astype(np.float32)
    B = rng.integers(-8, 9, (K, N)).astype(np.float32)
    bias = rng.integers(-100, 101, N).astype(np.float32)
    R = rng.integers(-100, 101, (batch, M, N)).astype(np.float32)
    C = np.zeros((batch, M, N), np.float32)
    orc.gemm_batched(0, 0, batch, M, N, K, A.reshape(-1), K, M * K, B.reshape(-1), N, 0,
                     C.reshape(-1), N, M * N, 0.5, bias, 0, R.reshape(-1), N, M * N)
    exact = 0.5 * np.einsum("bmk,kn->bmn", A.astype(np.int64), B.astype(np.int64)) + bias + R
    assert np.array_equal(C.astype(np.float64), exact)


def test_identity_epilogue_is_the_plain_gemm(orc):
    rng = np.random.default_rng(11)
    batch, M, N, K = 3, 17, 13, 40
    A = rng.standard_normal((batch, M, K)).astype(np.float32)
    B = rng.standard_normal((batch, K, N)).astype(np.float32)
    C = np.empty((batch, M, N), np.float32)
    orc.gemm_batched(0, 0, batch, M, N, K, A.reshape(-1), K, M * K, B.reshape(-1), N, K * N,
                     C.reshape(-1), N, M * N)
    for b in range(batch):
        assert np.array_equal(C[b].view(np.uint32), orc.gemm(A[b], B[b]).view(np.uint32))


def test_gelu_epilogue_is_the_elementwise_gelu(orc):
    rng = np.random.default_rng(12)
    A = rng.standard_normal((1, 20, 30)).astype(np.float32)
    B = rng.standard_normal((1, 30, 24)).astype(np.float32)
    bias = rng.standard_normal(24).astype(np.float32)
    C = np.empty((1, 20, 24), np.float32)
    orc.gemm_batched(0, 0, 1, 20, 24, 30, A.reshape(-1), 30, 0, B.reshape(-1), 24, 0,
                     C.reshape(-1), 24, 0, 1.0, bias, 1)
    y = (orc.gemm(A[0], B[0]) + bias).astype(np.float32)   # one rounding per add in float32
    assert np.array_equal(C[0].view(np.uint32), orc.gelu(y).view(np.uint32))


def test_empty_k_and_signed_zero_products(orc):
    # K = 0: acc = +0, so C = fl(alpha * +0): +0 for alpha > 0, -0 for alpha < 0,
    # then + bias exactly
    C = np.full(6, 7.0, np.float32)
    one = np.ones(1, np.float32)
    orc.gemm_batched(0, 0, 2, 1, 3, 0, one, 1, 0, one, 3, 0, C, 3, 3, -2.0)
    assert [fx.bits(float(v)) for v in C] == [0x80000000] * 6
    orc.gemm_batched(0, 0, 2, 1, 3, 0, one, 1, 0, one, 3, 0, C, 3, 3, 2.0)
    assert [fx.bits(float(v)) for v in C] == [0] * 6
    bias = np.array([1.5, -2.0, 0.25], np.float32)
    orc.gemm_batched(0, 0, 2, 1, 3, 0, one, 1, 0, one, 3, 0, C, 3, 3, 2.0, bias)
    assert np.array_equal(C, np.tile(bias, 2))
    # products that are all -0: +0 + (-0) = +0, and alpha = -1 turns it into -0
    A = np.zeros(4, np.float32)
    B = np.full(4, -3.0, np.float32)
    C = np.empty(1, np.float32)
    orc.gemm_batched(0, 0, 1, 1, 1, 4, A, 4, 0, B, 1, 0, C, 1, 0, -1.0)
    assert fx.bits(float(C[0])) == 0x80000000
