"""The parallel oracle helpers (tests/oracle_par.py) against the oracle run on
one thread: byte for byte the same results.

Every output element of the GEMM is one k-chain of its own ("Verde与RepOps"
§3.2) and every element of the mean + SGD one fold of its own ("Zoo Per-LLM
Chain Soundness" §5), so computing disjoint row or element ranges on separate
threads, with B handed over in column-major storage, must change no bit.  The
GPU parity tests compare the library with these helpers, so they are pinned
here to the single-threaded oracle.
"""
import numpy as np
import pytest

import oracle_par

F32 = np.float32


@pytest.mark.parametrize("M,N,K,bt", [(1, 1, 1, False), (67, 130, 45, False), (300, 257, 129, True),
                                      (97, 33, 700, True), (513, 64, 64, False)])
def test_parallel_gemm_equals_single_thread(orc, M, N, K, bt):
    rng = np.random.default_rng(M * 131 + N * 7 + K)
    A = rng.standard_normal((M, K)).astype(F32)
    B = rng.standard_normal((K, N)).astype(F32)
    Bv = np.asfortranarray(B) if bt else B
    want = orc.gemm(A, B)
    got = oracle_par.gemm(orc, A, Bv)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    rows = sorted(set(rng.integers(0, M, size=min(M, 9)).tolist()))
    cols = sorted(set(rng.integers(0, N, size=min(N, 7)).tolist()))
    sub = oracle_par.gemm(orc, A, Bv, rows=rows, cols=cols)
    assert np.array_equal(sub.view(np.uint32), want[np.ix_(rows, cols)].view(np.uint32))
    # any partition into parts gives the same bytes
    for parts in (1, 3, max(1, M)):
        assert np.array_equal(oracle_par.gemm(orc, A, Bv, parts=parts).view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("nC,n", [(1, 1), (3, 1000), (16, 200_003)])
def test_parallel_mean_sgd_equals_single_thread(orc, nC, n):
    rng = np.random.default_rng(nC * 1000 + n)
    grads = [(rng.standard_normal(n) * 1e-2).astype(F32) for _ in range(nC)]
    theta = (rng.standard_normal(n) * 0.02).astype(F32)
    order = [int(x) for x in rng.permutation(nC)]
    want = orc.mean_sgd(grads, order, 1e-3, theta)
    for lo, hi in ((0, n), (0, (n + 1) // 2), (n // 3, n)):
        got = oracle_par.mean_sgd(orc, grads, order, 1e-3, theta, lo, hi)
        assert np.array_equal(got.view(np.uint32), want[lo:hi].view(np.uint32)), (lo, hi)
