"""Reproducible (RepOps-style) operators for verifiable training on one GB300.

Python binding of librepops (include/repops.h): the functions here only
marshal torch CUDA tensors into pointers, sizes and strides and call the C ABI;
every operation runs in the library's CUDA kernels.  PyTorch provides device
memory and streams.

  gemm(A, B)                        order-fixed FP32 GEMM
                                    ("Verde与RepOps" §3.2, matmul example)
  sort_ids(ids)                     contributor order by DID bytes
  fixed_order_mean_sgd(...)         left-fold mean over contributors + SGD, in place
                                    ("Zoo Per-LLM Chain Soundness" §2, §5)
  merkle_sha256(t, leaf)            SHA-256 Merkle root of a tensor's bytes
                                    ("Zoo Per-LLM Chain Soundness" §1, §6, §7;
                                     "Verde与RepOps" §2.3.2)
"""
import ctypes

from . import _capi
from ._capi import (LOADER_AUTO, LOADER_CPASYNC, LOADER_TMA, MEAN_MAX_CONTRIBUTORS,
                    RepopsError, load)

__all__ = ["load", "version", "gemm", "gemm_config_count", "gemm_config_info",
           "gemm_auto_config", "sort_ids", "fixed_order_mean_sgd", "merkle_sha256",
           "merkle_workspace_bytes", "device_status", "RepopsError",
           "LOADER_AUTO", "LOADER_TMA", "LOADER_CPASYNC", "MEAN_MAX_CONTRIBUTORS"]


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def version() -> str:
    return load().repops_version().decode()


def _operand(X, name):
    """(pointer, leading dim, transposed) for a 2-D float32 CUDA view."""
    import torch
    if X.dtype != torch.float32 or X.dim() != 2 or not X.is_cuda:
        raise TypeError("%s must be a 2-D float32 CUDA tensor" % name)
    r, c = X.shape
    s0, s1 = X.stride()
    if s1 == 1 and s0 >= max(c, 1):
        return X.data_ptr(), s0, 0
    if s0 == 1 and s1 >= max(r, 1):
        return X.data_ptr(), s1, 1
    raise ValueError("%s must be row-major or a transposed (column-major) view" % name)


def gemm(A, B, out=None, *, config: int = -1, loader: int = LOADER_AUTO, stream=None):
    """C = A @ B with the order-fixed k-chain (bit-exact, no FMA).

    A: (M, K), B: (K, N) float32 CUDA tensors, row-major or transposed views.
    out: optional (M, N) float32 CUDA tensor with unit column stride."""
    import torch
    L = load()
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    pa, lda, ta = _operand(A, "A")
    pb, ldb, tb = _operand(B, "B")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if out.dtype != torch.float32 or out.dim() != 2 or tuple(out.shape) != (M, N) or \
            (N > 0 and out.stride(1) != 1):
        raise ValueError("out must be a (M, N) float32 tensor with unit column stride")
    ldc = max(out.stride(0), N, 1)
    rc = L.repops_gemm_f32_config(config, loader, ta, tb, M, N, K, pa, lda, pb, ldb,
                                  out.data_ptr(), ldc, _stream_handle(stream))
    _capi.check(rc, "repops_gemm_f32")
    return out


def gemm_raw(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, *, transA=0, transB=0,
             stream=None) -> int:
    """Direct call of repops_gemm_f32_ex on raw device pointers; returns the status."""
    return load().repops_gemm_f32_ex(transA, transB, M, N, K, A_ptr, lda, B_ptr, ldb,
                                     C_ptr, ldc, _stream_handle(stream))


def gemm_config_count() -> int:
    return load().repops_gemm_config_count()


def gemm_config_info(config: int) -> dict:
    v = [ctypes.c_int() for _ in range(5)]
    rc = load().repops_gemm_config_info(config, *[ctypes.byref(x) for x in v])
    _capi.check(rc, "repops_gemm_config_info")
    return dict(zip(("bm", "bn", "threads", "tm", "tn"), (x.value for x in v)))


def gemm_auto_config(M: int, N: int, K: int) -> int:
    return load().repops_gemm_auto_config(M, N, K)


def sort_ids(ids) -> list:
    """Contributor indices in unsigned lexicographic byte order of their IDs."""
    L = load()
    n = len(ids)
    blob = b"".join(ids)
    buf = ctypes.create_string_buffer(blob, max(len(blob), 1))
    lens = (ctypes.c_int64 * max(n, 1))(*[len(x) for x in ids])
    offs, o = [], 0
    for x in ids:
        offs.append(o)
        o += len(x)
    offs_c = (ctypes.c_int64 * max(n, 1))(*offs)
    order = (ctypes.c_int * max(n, 1))()
    rc = L.repops_sort_ids(n, ctypes.cast(buf, ctypes.c_void_p), ctypes.cast(offs_c, ctypes.c_void_p),
                           ctypes.cast(lens, ctypes.c_void_p), ctypes.cast(order, ctypes.c_void_p))
    _capi.check(rc, "repops_sort_ids")
    return [int(order[i]) for i in range(n)]


def fixed_order_mean_sgd(grads, order, eta: float, theta, *, stream=None):
    """theta -= eta * (left fold of grads in `order`) / len(grads), in place.

    grads: sequence of float32 CUDA tensors (or raw device pointers) with
    theta.numel() elements each; order: permutation of range(len(grads))."""
    L = load()
    nC = len(grads)
    ptrs = [g if isinstance(g, int) else g.data_ptr() for g in grads]
    for g in grads:
        if not isinstance(g, int) and g.numel() != theta.numel():
            raise ValueError("gradient and theta sizes differ")
    parr = (ctypes.c_void_p * max(nC, 1))(*ptrs)
    oarr = (ctypes.c_int * max(nC, 1))(*[int(x) for x in order])
    if len(order) != nC:
        raise ValueError("order must have one entry per contributor")
    rc = L.repops_fixed_order_mean_sgd(nC, theta.numel(), ctypes.cast(parr, ctypes.c_void_p),
                                       ctypes.cast(oarr, ctypes.c_void_p), ctypes.c_float(eta),
                                       theta.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_fixed_order_mean_sgd")
    return theta


def merkle_workspace_bytes(nbytes: int, leaf: int = 4096) -> int:
    return load().repops_merkle_workspace_bytes(nbytes, leaf)


def merkle_sha256(t, leaf: int = 4096, out=None, *, nbytes: int = None, workspace=None,
                  stream=None):
    """32-byte SHA-256 Merkle root (uint8 CUDA tensor) of the bytes of `t`.

    t: a contiguous CUDA tensor; its storage bytes are hashed as stored.
    nbytes: hash only the first nbytes bytes.  workspace: optional uint8 CUDA
    tensor used as scratch instead of a stream-ordered allocation."""
    import torch
    L = load()
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("t must be a contiguous CUDA tensor")
    n = t.numel() * t.element_size() if nbytes is None else int(nbytes)
    if out is None:
        out = torch.empty(32, dtype=torch.uint8, device=t.device)
    s = _stream_handle(stream)
    if workspace is None:
        rc = L.repops_merkle_sha256(t.data_ptr(), n, leaf, out.data_ptr(), s)
    else:
        rc = L.repops_merkle_sha256_ws(t.data_ptr(), n, leaf, out.data_ptr(), workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(), s)
    _capi.check(rc, "repops_merkle_sha256")
    return out


def device_status(stream=None) -> int:
    """Synchronises the stream; returns and clears the sticky device status."""
    v = ctypes.c_int(0)
    rc = load().repops_device_status(_stream_handle(stream), ctypes.byref(v))
    _capi.check(rc, "repops_device_status")
    return v.value
