"""GPU test of the boundary's thread safety (include/repops.h conventions:
any host thread may call any entry point).

Four host threads, each on its own CUDA stream with its own status word, run
the hot path over and over at the same time: a ragged GEMM with a transposed
B (operand copy into pool scratch), a GEMM on the chained k-split (partial-sum
scratch and flags), the mean + SGD and a Merkle root.  The library's host
code runs concurrently (ctypes releases the GIL): the per-device caches, the
scratch pool and the status words are shared state.  Every result must be the
oracle's and every thread's status word must stay clear.
"""
import threading

import numpy as np
import pytest
import torch

import oracle_par
from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
THREADS = 4
ROUNDS = 6


def u32(x):
    return np.ascontiguousarray(x).view(np.uint32)


def test_concurrent_callers_get_the_oracle_bits(rp, orc):
    # shared inputs (read only) and the expected results, from the oracle
    A = inputs.normal((700, 900), 1.0, 61, DEV)
    Bt = inputs.normal((1500, 900), 1.0, 62, DEV)          # B = Bt^T, stored transposed
    A2 = inputs.normal((2048, 1024), 1.0, 63, DEV)
    B2 = inputs.normal((1024, 2048), 1.0, 64, DEV)
    rows2 = list(range(0, 2048, 61)) + [2047]
    want1 = u32(oracle_par.gemm(orc, A, Bt.t()))
    want2 = u32(oracle_par.gemm(orc, A2, B2, rows=rows2))
    n, nC = 1_000_003, 5
    grads = [inputs.normal((n,), 1e-2, 70 + r, DEV) for r in range(nC)]
    theta0 = inputs.normal((n,), 0.02, 69, DEV)
    order = rp.sort_ids(inputs.contributor_ids(nC, 71))
    want_theta = orc.mean_sgd([g.cpu().numpy() for g in grads], order, 1e-3, theta0.cpu().numpy())
    T = inputs.normal((3 << 18,), 0.02, 72, DEV)
    want_root = orc.merkle_root(T.cpu().numpy(), 4096)
    torch.cuda.synchronize()

    errors = []

    def caller(t):
        try:
            torch.cuda.set_device(0)
            word = torch.zeros(1, dtype=torch.int32, device=DEV)
            rp.set_thread_status_word(word)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                theta = theta0.clone()
                for it in range(ROUNDS):
                    C1 = rp.gemm(A, Bt.t())
                    C2 = rp.gemm(A2, B2)
                    if it == 0:
                        rp.fixed_order_mean_sgd(grads, order, 1e-3, theta)
                    root = rp.merkle_sha256(T)
                    s.synchronize()
                    if not np.array_equal(u32(C1.cpu().numpy()), want1):
                        errors.append((t, it, "gemm transposed B"))
                    if not np.array_equal(u32(C2[rows2].cpu().numpy()), want2):
                        errors.append((t, it, "gemm chained"))
                    if bytes(root.cpu().numpy()) != want_root:
                        errors.append((t, it, "merkle"))
                    if it == 0 and not np.array_equal(u32(theta.cpu().numpy()), u32(want_theta)):
                        errors.append((t, it, "mean+sgd"))
                if rp.device_status(s) != 0:
                    errors.append((t, "status"))
            rp.set_thread_status_word(None)
        except Exception as e:   # reported below, on the main thread
            errors.append((t, repr(e)))

    ths = [threading.Thread(target=caller, args=(t,)) for t in range(THREADS)]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    assert not errors, errors
    assert rp.device_status() == 0
