"""GPU tests of the library's scratch pool (repops_scratch_set_keep_bytes,
repops_scratch_release, repops_scratch_reserved_bytes; "Scratch memory" in
include/repops.h).

By default the library holds no memory between calls: scratch taken by a call
is handed back at the next synchronisation.  When the caller asks for it, the
pool keeps freed scratch mapped across synchronisations (so the next call does
not map it again) until a release.  The device's default pool is neither used
nor changed, and the bits are the oracle's in every mode.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle_par
from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def default_pool_release_threshold() -> int:
    cu = ctypes.CDLL("libcuda.so.1")
    d = ctypes.c_int()
    assert cu.cuDeviceGet(ctypes.byref(d), torch.cuda.current_device()) == 0
    pool = ctypes.c_void_p()
    assert cu.cuDeviceGetDefaultMemPool(ctypes.byref(pool), d) == 0
    v = ctypes.c_uint64()
    assert cu.cuMemPoolGetAttribute(pool, 4, ctypes.byref(v)) == 0   # release threshold
    return v.value


def bits(t):
    return t.cpu().numpy().view(np.uint32)


def test_scratch_kept_only_when_asked_and_until_released(rp, orc):
    # 1000 x 1001 x 520 with B stored transposed (1.04 GFLOP): B is copied
    # into a row-major scratch copy before the kernel runs
    A = inputs.normal((1000, 520), 1.0, 41, DEV)
    B = inputs.normal((1001, 520), 1.0, 42, DEV).t()
    want = oracle_par.gemm(orc, A, B).view(np.uint32)
    threshold = default_pool_release_threshold()
    results = []

    def gemm_pool():
        # the C entry point itself (the binding's gemm passes a workspace instead)
        C = torch.empty((1000, 1001), device=DEV)
        assert rp.gemm_raw(1000, 1001, 520, A.data_ptr(), 520, B.data_ptr(), 520, C.data_ptr(), 1001,
                           transB=1) == 0
        return C

    try:
        # default: nothing held once the call's work has been synchronised
        results.append(gemm_pool())
        torch.cuda.synchronize()
        assert rp.scratch_reserved_bytes() == 0
        # kept on request, across synchronisations, until released
        rp.scratch_set_keep_bytes(1 << 30)
        for _ in range(2):
            results.append(gemm_pool())
            torch.cuda.synchronize()
            assert rp.scratch_reserved_bytes() >= 1001 * 520 * 4
        rp.scratch_release()
        torch.cuda.synchronize()
        assert rp.scratch_reserved_bytes() == 0
        results.append(gemm_pool())
        torch.cuda.synchronize()
        assert rp.scratch_reserved_bytes() >= 1001 * 520 * 4
    finally:
        rp.scratch_set_keep_bytes(0)
        rp.scratch_release()
    torch.cuda.synchronize()
    assert rp.scratch_reserved_bytes() == 0
    for C in results:
        assert np.array_equal(bits(C), want)
    assert default_pool_release_threshold() == threshold


def test_scratch_shared_by_streams_and_entry_points(rp, orc):
    # a chained-split GEMM, a Merkle root and a transposed-B GEMM on two
    # streams, over and over, with releases in between: every result the
    # oracle's
    A = inputs.normal((2048, 2048), 1.0, 43, DEV)
    B = inputs.normal((2048, 2048), 1.0, 44, DEV)
    T = inputs.normal((1 << 20,), 0.02, 45, DEV)
    rows = list(range(0, 2048, 97))
    want_rows = oracle_par.gemm(orc, A, B, rows=rows)
    want_root = orc.merkle_root(T.cpu().numpy(), 4096)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    rp.scratch_set_keep_bytes(256 << 20)
    for it in range(4):
        with torch.cuda.stream(s1):
            C = rp.gemm(A, B)
        with torch.cuda.stream(s2):
            C2 = rp.gemm(A, B.t().contiguous().t())
            root = rp.merkle_sha256(T)
        torch.cuda.synchronize()
        for X in (C, C2):
            assert np.array_equal(X[rows].cpu().numpy().view(np.uint32), want_rows.view(np.uint32)), it
        assert bytes(root.cpu().numpy()) == want_root, it
        if it % 2:
            rp.scratch_release()
    rp.scratch_set_keep_bytes(0)
    rp.scratch_release()
    assert rp.device_status() == 0


@pytest.mark.parametrize("M,N,K,tb", [(2048, 2048, 2048, False), (1536, 1536, 1536, True), (4097, 1024, 3000, False),
                                      (300, 200, 100, False)])
def test_gemm_caller_workspace(rp, orc, M, N, K, tb):
    # repops_gemm_workspace_bytes sizes the automatic plan's scratch (operand
    # copies, chained-split sums); repops_gemm_f32_ws takes it from the
    # caller's buffer: the same bits, and nothing from the library's pool
    L = rp.load()
    A = inputs.normal((M, K), 1.0, 51, DEV)
    B = inputs.normal((N, K), 1.0, 52, DEV).t() if tb else inputs.normal((K, N), 1.0, 52, DEV)
    ldb = B.stride(1) if tb else B.stride(0)
    need = L.repops_gemm_workspace_bytes(0, int(tb), M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), ldb)
    if M * N <= 196_608 or 2.0 * M * N * K < 1e9:
        assert need == 0
    else:
        assert need > 0
    rows = list(range(0, M, max(1, M // 17))) + [M - 1]
    want = oracle_par.gemm(orc, A, B, rows=rows).view(np.uint32)
    s = torch.cuda.current_stream().cuda_stream
    try:
        rp.scratch_set_keep_bytes(1 << 30)
        rp.scratch_release()
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=DEV)
        C = torch.full((M, N), float("nan"), device=DEV)
        assert L.repops_gemm_f32_ws(0, int(tb), M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), ldb, C.data_ptr(),
                                    N, ws.data_ptr(), need, s) == 0
        torch.cuda.synchronize()
        assert rp.scratch_reserved_bytes() == 0                     # the pool was not used
        assert np.array_equal(C[rows].cpu().numpy().view(np.uint32), want)
        C2 = rp.gemm(A, B)                                           # the binding passes a workspace too
        torch.cuda.synchronize()
        assert rp.scratch_reserved_bytes() == 0
        assert torch.equal(C2.view(torch.int32), C.view(torch.int32))
        if need:
            # a workspace one byte short is not used: the scratch comes from the pool
            C3 = torch.full((M, N), float("nan"), device=DEV)
            assert L.repops_gemm_f32_ws(0, int(tb), M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), ldb,
                                        C3.data_ptr(), N, ws.data_ptr(), need - 1, s) == 0
            torch.cuda.synchronize()
            assert rp.scratch_reserved_bytes() > 0
            assert torch.equal(C3.view(torch.int32), C.view(torch.int32))
            # misaligned or overlapping workspaces are refused before any launch
            assert L.repops_gemm_f32_ws(0, int(tb), M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), ldb,
                                        C3.data_ptr(), N, ws.data_ptr() + 16, need, s) == -1
            assert L.repops_gemm_f32_ws(0, int(tb), M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), ldb,
                                        C3.data_ptr(), N, C3.data_ptr(), need, s) == -2
    finally:
        rp.scratch_set_keep_bytes(0)
        rp.scratch_release()
    assert rp.device_status() == 0
