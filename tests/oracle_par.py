"""Test helper: the oracle over disjoint parts of a problem, on every host core.

Every output element of the oracle's GEMM is one k-chain of its own, and
every element of its mean + SGD one fold of its own, so computing disjoint
row ranges (or element ranges) on separate threads changes no operation of
any element: the result is the single-threaded oracle's, byte for byte.
ctypes releases the GIL while the C oracle runs, so plain threads use every
core.  B is handed to the oracle's GEMM in column-major storage (the same
logical matrix) so each k-chain reads both operands at unit stride.
"""
import concurrent.futures as cf
import os

import numpy as np


def host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _np(x) -> np.ndarray:
    """float32 numpy copy of a (possibly device, possibly strided) torch tensor
    or array, in row-major storage."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def gemm(orc, A, B, rows=None, cols=None, parts=None):
    """Oracle A @ B restricted to `rows` x `cols` (index lists; None = all),
    as a float32 array of shape (len(rows), len(cols)).

    A is split into row blocks, one per task."""
    An = _np(A)
    Bn = np.asfortranarray(_np(B))
    if rows is not None:
        An = np.ascontiguousarray(An[np.asarray(rows)])
    if cols is not None:
        Bn = np.asfortranarray(Bn[:, np.asarray(cols)])
    M, N = An.shape[0], Bn.shape[1]
    out = np.empty((M, N), dtype=np.float32)
    if M == 0 or N == 0:
        return out
    nparts = parts or min(M, 4 * host_cores())
    cuts = [M * p // nparts for p in range(nparts + 1)]

    def part(p):
        r0, r1 = cuts[p], cuts[p + 1]
        if r1 > r0:
            orc.gemm(An[r0:r1], Bn, out=out[r0:r1])

    with cf.ThreadPoolExecutor(max_workers=host_cores()) as ex:
        list(ex.map(part, range(nparts)))
    return out


def mean_sgd(orc, grads, order, eta, theta, lo, hi):
    """Oracle theta - eta * mean over elements [lo, hi) of host arrays, split
    into element ranges across the cores."""
    n = hi - lo
    out = np.empty(n, dtype=np.float32)
    nparts = min(max(n // 65536, 1), 4 * host_cores())
    cuts = [lo + n * p // nparts for p in range(nparts + 1)]

    def part(p):
        a, b = cuts[p], cuts[p + 1]
        if b > a:
            out[a - lo:b - lo] = orc.mean_sgd([g[a:b] for g in grads], order, eta, theta[a:b])

    with cf.ThreadPoolExecutor(max_workers=host_cores()) as ex:
        list(ex.map(part, range(nparts)))
    return out
