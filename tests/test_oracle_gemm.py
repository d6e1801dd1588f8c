"""Pins the GEMM oracle to things other than itself.

The method: "Verde与RepOps" §3.2 matmul example -- C[i][j] = sum over k of
A[i][k]*B[k][j], k strictly increasing from 0, each product and each sum
rounded to binary32 (no FMA: "Zoo Per-LLM Chain Soundness" §5).
"""
import numpy as np
import pytest

import fp32_exact as fx


def _f32bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def test_fp_environment(orc):
    assert orc.lib().oracle_fp_env_ok() == 1


@pytest.mark.parametrize("M,N,K", [(7, 9, 1), (13, 5, 64), (17, 33, 4096), (1, 1, 4096)])
def test_integer_inputs_give_the_exact_sum(orc, M, N, K):
    # |partial sums| <= 64*4096 < 2^24: every product and sum is exact, so the
    # result is the integer matrix product, whatever the order.
    rng = np.random.default_rng(M * 1000 + K)
    A = rng.integers(-8, 9, size=(M, K))
    B = rng.integers(-8, 9, size=(K, N))
    want = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
    got = orc.gemm(A.astype(np.float32), B.astype(np.float32))
    assert np.array_equal(_f32bits(got), _f32bits(want))


def _wide_floats(rng, shape):
    # values spread over many binades, with both signs, some exact zeros
    mant = rng.uniform(-1, 1, size=shape)
    expo = rng.integers(-30, 30, size=shape)
    v = (mant * np.exp2(expo)).astype(np.float32)
    v[rng.random(shape) < 0.05] = 0.0
    return v


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 4, 5), (8, 8, 8), (2, 3, 64), (5, 2, 33)])
def test_brute_force_exact_rational(orc, M, N, K):
    rng = np.random.default_rng(17 + M + 10 * N + 100 * K)
    A = _wide_floats(rng, (M, K))
    B = _wide_floats(rng, (K, N))
    got = orc.gemm(A, B)
    for i in range(M):
        for j in range(N):
            want = fx.gemm_entry(A[i, :].tolist(), B[:, j].tolist())
            assert fx.bits(float(got[i, j])) == fx.bits(want), (i, j)


def test_numpy_scalar_loop(orc):
    # numpy float32 scalar ops round each result to binary32 on their own
    rng = np.random.default_rng(5)
    A = rng.standard_normal((4, 40)).astype(np.float32)
    B = rng.standard_normal((40, 3)).astype(np.float32)
    got = orc.gemm(A, B)
    for i in range(4):
        for j in range(3):
            s = np.float32(0.0)
            for k in range(40):
                p = np.float32(A[i, k] * B[k, j])
                s = np.float32(s + p)
            assert _f32bits(s) == _f32bits(got[i, j])


def test_order_detector(orc, golden):
    case = golden["gemm_order_detector"]
    a = np.array(case["a_row"], dtype=np.float32)
    b = np.array(case["b_col"], dtype=np.float32)
    got = orc.gemm(a[None, :], b[:, None])
    assert int(_f32bits(got)[0, 0]) == int(case["expected_bits"], 16)
    for ob in case["other_orders_bits"]:
        assert int(_f32bits(got)[0, 0]) != int(ob, 16)
    # planted into a random row of a larger problem
    rng = np.random.default_rng(3)
    A = rng.integers(-3, 4, size=(6, 4)).astype(np.float32)
    A[4] = a
    B = np.ones((4, 5), dtype=np.float32)
    C = orc.gemm(A, B)
    assert np.all(_f32bits(C[4]) == int(case["expected_bits"], 16))


def test_fma_detector(orc, golden):
    case = golden["gemm_fma_detector"]
    a = np.array([int(x, 16) for x in case["a_row_bits"]], dtype=np.uint32).view(np.float32)
    b = np.array([int(x, 16) for x in case["b_col_bits"]], dtype=np.uint32).view(np.float32)
    got = orc.gemm(a[None, :], b[:, None])
    assert int(_f32bits(got)[0, 0]) == int(case["expected_bits"], 16)
    assert int(_f32bits(got)[0, 0]) != int(case["fma_bits"], 16)


def test_k_order_is_increasing(orc):
    # Only increasing k reproduces the order detector when it is reversed in
    # storage: reversing the k axis of both operands must change the bits.
    a = np.array([1.0, -1e8, 1.0, 1e8], dtype=np.float32)   # reversed detector
    C = orc.gemm(a[None, :], np.ones((4, 1), np.float32))
    # increasing k on the reversed row: 1-1e8 -> -1e8, +1 -> -1e8, +1e8 -> 0
    assert int(_f32bits(C)[0, 0]) == 0


def test_zero_k_writes_positive_zero(orc):
    A = np.zeros((3, 0), np.float32)
    B = np.zeros((0, 4), np.float32)
    C = np.full((3, 4), np.nan, np.float32)
    orc.gemm(A, B, out=C)
    assert np.all(_f32bits(C) == 0)


def test_result_is_never_negative_zero(orc):
    # products that are -0 or cancel exactly leave the +0 start in place
    A = np.array([[-0.0, -0.0, 2.0, -2.0]], np.float32)
    B = np.array([[1.0], [3.0], [1.0], [1.0]], np.float32)
    C = orc.gemm(A, B)
    assert int(_f32bits(C)[0, 0]) == 0


def test_subnormal_products_are_kept(orc):
    t = np.float32(2.0 ** -70)
    A = np.array([[t, t]], np.float32)
    B = np.array([[t], [t]], np.float32)
    C = orc.gemm(A, B)
    # 2^-140 + 2^-140 = 2^-139, both subnormal: no flush to zero
    assert float(C[0, 0]) == 2.0 ** -139


def test_k_equals_one_is_the_elementwise_outer_product(orc):
    rng = np.random.default_rng(11)
    a = rng.standard_normal(9).astype(np.float32)
    b = rng.standard_normal(7).astype(np.float32)
    C = orc.gemm(a[:, None], b[None, :])
    want = np.multiply.outer(a, b)     # float32 multiply, one rounding each
    # + 0.0 does not change a nonzero value, and turns -0 into +0
    want = want + np.float32(0.0)
    assert np.array_equal(_f32bits(C), _f32bits(want))


def test_storage_layout_does_not_change_bits(orc):
    rng = np.random.default_rng(23)
    A = rng.standard_normal((37, 53)).astype(np.float32)
    B = rng.standard_normal((53, 29)).astype(np.float32)
    C0 = orc.gemm(A, B)
    At = np.ascontiguousarray(A.T).T          # column-major storage of A
    Bt = np.ascontiguousarray(B.T).T          # column-major storage of B
    assert np.array_equal(_f32bits(orc.gemm(At, B)), _f32bits(C0))
    assert np.array_equal(_f32bits(orc.gemm(A, Bt)), _f32bits(C0))
    assert np.array_equal(_f32bits(orc.gemm(At, Bt)), _f32bits(C0))
    # padded leading dimensions
    Ap = np.zeros((37, 64), np.float32); Ap[:, :53] = A
    Bp = np.zeros((53, 40), np.float32); Bp[:, :29] = B
    assert np.array_equal(_f32bits(orc.gemm(Ap[:, :53], Bp[:, :29])), _f32bits(C0))


def test_row_blocks_match_full_product(orc):
    # any order over i and j: computing row and column blocks separately is the
    # same computation element by element
    rng = np.random.default_rng(29)
    A = rng.standard_normal((20, 31)).astype(np.float32)
    B = rng.standard_normal((31, 18)).astype(np.float32)
    C = orc.gemm(A, B)
    C2 = np.empty_like(C)
    for i0 in range(0, 20, 7):
        for j0 in range(0, 18, 5):
            C2[i0:i0 + 7, j0:j0 + 5] = orc.gemm(A[i0:i0 + 7], B[:, j0:j0 + 5])
    assert np.array_equal(_f32bits(C), _f32bits(C2))
