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
  merkle_tree / merkle_proof /      whole tree, inclusion proofs, membership check
  merkle_verify                     ("Verde与RepOps" §2.4)
  replay(...)                       mean + SGD + commit per block, in order
                                    ("Zoo Per-LLM Chain Soundness" §7)
  softmax_rows / layernorm_rows /   order-fixed row operators and GeLU
  rmsnorm_rows / gelu               ("Verde与RepOps" §3.2, §4.3)
  gemm_batched(A, B, ...)           batched GEMM with a fused epilogue
                                    (alpha, bias, GeLU, residual)
  convert / gemm_typed              binary16 / bfloat16 storage around the
                                    binary32 path ("Verde与RepOps" §3.3, §5.3)
  rolling_hash(words, window)       Rabin-Karp hashes of uint32 batch rows (ZKDV)
  colsum / gelu_backward /          backward operators of a training step
  rmsnorm_backward / softmax_backward
  swiglu / swiglu_backward /        SiLU-gated MLP activation and rotary
  rope_frequencies / rope_table /   position embeddings of a Llama-style layer
  rope                              ("Verde与RepOps" §4.3)
  host_empty(shape, dtype)          page-locked host memory in huge pages for the
                                    host-buffer calls (gemm_host, ..._host)
"""
import ctypes

from . import _capi
from ._capi import (ACT_GELU, ACT_NONE, LOADER_AUTO, LOADER_CPASYNC, LOADER_DIRECT, LOADER_TMA,
                    MEAN_MAX_CONTRIBUTORS, TYPE_BF16, TYPE_F16, TYPE_F32, RepopsError, load)

__all__ = ["load", "version", "scratch_set_keep_bytes", "scratch_release", "scratch_reserved_bytes", "host_empty", "gemm", "gemm_chained", "gemm_auto_chained", "fixed_order_mean_sgd_host", "merkle_sha256_host", "attention_causal", "gemm_config_occupancy", "gemm_host", "gemm_config_count", "gemm_config_info",
           "gemm_auto_config", "gemm_small_output", "sha256_rate_probe", "sort_ids", "fixed_order_mean_sgd", "merkle_sha256",
           "merkle_workspace_bytes", "merkle_tree", "merkle_proof", "merkle_verify", "replay",
           "softmax_rows", "layernorm_rows", "rmsnorm_rows", "gelu", "gemm_batched",
           "convert", "gemm_typed", "rolling_hash", "TYPE_F32", "TYPE_F16", "TYPE_BF16",
           "colsum", "gelu_backward", "rmsnorm_backward", "softmax_backward",
           "swiglu", "swiglu_backward", "rope_frequencies", "rope_table", "rope",
           "device_status", "set_thread_status_word", "RepopsError", "ACT_NONE", "ACT_GELU",
           "LOADER_AUTO", "LOADER_TMA", "LOADER_CPASYNC", "LOADER_DIRECT", "MEAN_MAX_CONTRIBUTORS"]


# Outputs the functions below allocate come from torch's caching allocator on
# the current stream; a caller passing another `stream` must keep them alive
# (or record them on that stream) until that stream has finished with them.
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
    if config < 0 and loader == LOADER_AUTO:
        # the automatic choice's scratch comes from torch's caching allocator
        # (repops_gemm_f32_ws), so nothing is mapped afresh after a sync
        need = L.repops_gemm_workspace_bytes(ta, tb, M, N, K, pa, lda, pb, ldb)
        ws = _workspace(need, A.device, stream) if need else None
        if ws is not None:
            rc = L.repops_gemm_f32_ws(ta, tb, M, N, K, pa, lda, pb, ldb, out.data_ptr(), ldc, ws.data_ptr(),
                                      need, _stream_handle(stream))
            _capi.check(rc, "repops_gemm_f32_ws")
            return out
    rc = L.repops_gemm_f32_config(config, loader, ta, tb, M, N, K, pa, lda, pb, ldb,
                                  out.data_ptr(), ldc, _stream_handle(stream))
    _capi.check(rc, "repops_gemm_f32")
    return out


def _workspace(nbytes, device, stream):
    """A byte buffer from torch's caching allocator for a call on `stream`,
    kept from reuse until that stream's work is done; None when the stream is
    a raw handle the allocator cannot track (the library's pool is used)."""
    import torch
    if isinstance(stream, int):
        return None
    ws = torch.empty(int(nbytes), dtype=torch.uint8, device=device)
    if stream is not None and stream != torch.cuda.current_stream(device):
        ws.record_stream(stream)
    return ws


def gemm_chained(A, B, out=None, *, config: int = -1, workers: int = 0, stream=None):
    """C = A @ B on the chained k-split schedule (repops_gemm_f32_chained):
    `workers` persistent CTAs, a tile's k-chain possibly continued by the next
    worker; the same bits as gemm()."""
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
    rc = L.repops_gemm_f32_chained(config, workers, ta, tb, M, N, K, pa, lda, pb, ldb,
                                   out.data_ptr(), ldc, _stream_handle(stream))
    _capi.check(rc, "repops_gemm_f32_chained")
    return out


def _batched_operand(X, name):
    """(pointer, leading dim, batch stride, transposed, batch) of a float32 CUDA
    tensor of shape (batch, rows, cols), or (rows, cols) shared by all batches.
    Each matrix must be row-major or a transposed view; the batch stride is
    whatever the tensor's first stride is (0 for an expanded tensor)."""
    import torch
    if X.dtype != torch.float32 or X.dim() not in (2, 3) or not X.is_cuda:
        raise TypeError("%s must be a 2-D or 3-D float32 CUDA tensor" % name)
    if X.dim() == 2:
        p, ld, t = _operand(X, name)
        return p, ld, 0, t, None
    b, r, c = X.shape
    sb, s0, s1 = X.stride()
    if s1 == 1 and s0 >= max(c, 1):
        return X.data_ptr(), s0, sb, 0, b
    if s0 == 1 and s1 >= max(r, 1):
        return X.data_ptr(), s1, sb, 1, b
    raise ValueError("%s: each matrix must be row-major or a transposed view" % name)


def gemm_batched(A, B, out=None, *, alpha: float = 1.0, bias=None, act: int = ACT_NONE,
                 residual=None, causal_first: int = -1, k_lo: int = -1, k_hi: int = -1, config: int = -1,
                 loader: int = LOADER_AUTO, stream=None):
    """out[b] = epilogue(A[b] @ B[b]) with the order-fixed k-chain, then
    y = alpha*acc, + bias[j], GeLU (act=ACT_GELU), + residual[b][i][j], each one
    binary32 rounding (repops_gemm_f32_batched).

    A: (batch, M, K) or (M, K) shared; B: (batch, K, N), (K, N) shared, or
    (batch / g, K, N) with each B shared by g consecutive batches (the query
    heads of a grouped-query attention group and their key/value head); every
    matrix row-major or a transposed view, batches at any stride (attention
    heads as column blocks: X.view(T, H, d).transpose(0, 1)).  out: (batch, M,
    N) or (M, N), unit column stride, batches stacked or interleaved.
    residual: shaped like out; may be out itself.  bias: (N,) contiguous.
    causal_first >= 0: elements with j > causal_first + i are left unspecified
    (whole tiles above that boundary are skipped).  k_lo / k_hi >= 0: row i's
    k-chain covers [i - k_lo, i + k_hi] only (A must be +-0 outside that band
    and B finite: see repops_gemm_f32_batched)."""
    import torch
    L = load()
    pa, lda, sa, ta, ba = _batched_operand(A, "A")
    pb, ldb, sb, tb, bb = _batched_operand(B, "B")
    M, K = A.shape[-2:]
    K2, N = B.shape[-2:]
    if K != K2:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    group = 1
    if ba is not None and bb is not None and ba != bb:
        if bb == 0 or ba % bb:
            raise ValueError("B's batch count must equal A's or divide it")
        group = ba // bb
    batch = ba if ba is not None else bb
    if out is None:
        shape = (M, N) if batch is None else (batch, M, N)
        out = torch.empty(shape, dtype=torch.float32, device=A.device)
    nb = 1 if batch is None else batch
    if out.dtype != torch.float32 or tuple(out.shape[-2:]) != (M, N) or \
            out.dim() != (2 if batch is None else 3) or (batch is not None and out.shape[0] != batch) or \
            (N > 0 and out.stride(-1) != 1):
        raise ValueError("out must be a float32 tensor of shape %s with unit column stride"
                         % (((M, N) if batch is None else (batch, M, N)),))
    ldc = max(out.stride(-2), N, 1)
    sc = out.stride(0) if batch is not None else 0
    pr, ldr, sr = None, 0, 0
    if residual is not None:
        if residual.dtype != torch.float32 or residual.shape != out.shape or \
                (N > 0 and residual.stride(-1) != 1):
            raise ValueError("residual must be shaped like out, float32, unit column stride")
        pr, ldr = residual.data_ptr(), max(residual.stride(-2), N, 1)
        sr = residual.stride(0) if batch is not None else 0
    pbias = None
    if bias is not None:
        if bias.dtype != torch.float32 or bias.dim() != 1 or bias.numel() != N or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous float32 vector of N values")
        pbias = bias.data_ptr()
    rc = L.repops_gemm_f32_batched(config, loader, ta, tb, nb, M, N, K, pa, lda, sa, pb, ldb, sb,
                                   out.data_ptr(), ldc, sc, ctypes.c_float(alpha), pbias, int(act),
                                   pr, ldr, sr, int(causal_first), int(k_lo), int(k_hi), group,
                                   _stream_handle(stream))
    _capi.check(rc, "repops_gemm_f32_batched")
    return out


def gemm_host(A, B, out=None, *, stream=None):
    """C = A @ B for row-major float32 CPU tensors (pin them for full speed):
    the copies to and from the device overlap the GEMM's row blocks
    (repops_gemm_f32_host).  Asynchronous on `stream`: synchronise it before
    reading `out`; A, B and out must stay alive until then."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    for t, n in ((A, "A"), (B, "B")):
        if t.dtype != torch.float32 or t.is_cuda or t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
            raise ValueError("%s must be a row-major float32 CPU tensor" % n)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, pin_memory=A.is_pinned())
    if out.dtype != torch.float32 or out.is_cuda or tuple(out.shape) != (M, N) or (N > 1 and out.stride(1) != 1):
        raise ValueError("out must be a row-major (M, N) float32 CPU tensor")
    rc = load().repops_gemm_f32_host(M, N, K, A.data_ptr(), max(A.stride(0), K, 1), B.data_ptr(),
                                     max(B.stride(0), N, 1), out.data_ptr(), max(out.stride(0), N, 1),
                                     _stream_handle(stream))
    _capi.check(rc, "repops_gemm_f32_host")
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


def gemm_config_occupancy(config: int) -> int:
    """Resident CTAs per SM of a configuration's TMA kernel on the current device."""
    rc = load().repops_gemm_config_occupancy(config)
    _capi.check(rc if rc < 0 else 0, "repops_gemm_config_occupancy")
    return rc


def gemm_auto_config(M: int, N: int, K: int) -> int:
    return load().repops_gemm_auto_config(M, N, K)


def gemm_auto_chained(M: int, N: int, K: int) -> bool:
    """True when the automatic choice runs M x N x K on the chained k-split."""
    return bool(load().repops_gemm_auto_chained(M, N, K))


def gemm_small_output(M: int, N: int, K: int) -> bool:
    """True when the automatic GEMM runs M x N x K on the small-output kernel."""
    return bool(load().repops_gemm_small_output(M, N, K))


def sha256_rate_probe(threads: int, iters: int, out=None, stream=None):
    """(threads, 8) int32 tensor of SHA-256 state words: thread t's digest of
    its 64-byte block (big-endian words 16t .. 16t + 15) repeated `iters`
    times, computed with the message in registers (repops_sha256_rate_probe,
    the Merkle kernels' compression-rate ceiling)."""
    import torch
    if out is None:
        out = torch.empty((threads, 8), dtype=torch.int32, device="cuda")
    if out.dtype != torch.int32 or not out.is_contiguous() or out.numel() != 8 * threads:
        raise ValueError("out must be a contiguous int32 tensor of threads x 8 words")
    rc = load().repops_sha256_rate_probe(threads, iters, out.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_sha256_rate_probe")
    return out


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


def _storage_type(dtype):
    import torch
    t = {torch.float32: TYPE_F32, torch.float16: TYPE_F16, torch.bfloat16: TYPE_BF16}.get(dtype)
    if t is None:
        raise TypeError("storage type must be float32, float16 or bfloat16, not %s" % dtype)
    return t


def fixed_order_mean_sgd(grads, order, eta: float, theta, *, grad_dtype=None, stream=None):
    """theta -= eta * (left fold of grads in `order`) / len(grads), in place.

    grads: sequence of CUDA tensors (or raw device pointers) with theta.numel()
    elements each, stored as float32, float16 or bfloat16 (widened exactly;
    theta stays float32); order: permutation of range(len(grads)).
    grad_dtype: the gradients' dtype when they are raw pointers."""
    L = load()
    nC = len(grads)
    dts = {g.dtype for g in grads if not isinstance(g, int)}
    if grad_dtype is not None:
        dts.add(grad_dtype)
    if len(dts) > 1:
        raise TypeError("gradients of different dtypes")
    gtype = _storage_type(dts.pop()) if dts else TYPE_F32
    ptrs = [g if isinstance(g, int) else g.data_ptr() for g in grads]
    for g in grads:
        if not isinstance(g, int) and g.numel() != theta.numel():
            raise ValueError("gradient and theta sizes differ")
    parr = (ctypes.c_void_p * max(nC, 1))(*ptrs)
    oarr = (ctypes.c_int * max(nC, 1))(*[int(x) for x in order])
    if len(order) != nC:
        raise ValueError("order must have one entry per contributor")
    if gtype == TYPE_F32:
        rc = L.repops_fixed_order_mean_sgd(nC, theta.numel(), ctypes.cast(parr, ctypes.c_void_p),
                                           ctypes.cast(oarr, ctypes.c_void_p), ctypes.c_float(eta),
                                           theta.data_ptr(), _stream_handle(stream))
        _capi.check(rc, "repops_fixed_order_mean_sgd")
    else:
        rc = L.repops_fixed_order_mean_sgd_typed(nC, theta.numel(), ctypes.cast(parr, ctypes.c_void_p), gtype,
                                                 ctypes.cast(oarr, ctypes.c_void_p), ctypes.c_float(eta),
                                                 theta.data_ptr(), _stream_handle(stream))
        _capi.check(rc, "repops_fixed_order_mean_sgd_typed")
    return theta


def fixed_order_mean_sgd_host(grads, order, eta: float, theta, *, stream=None):
    """fixed_order_mean_sgd on float32 CPU tensors (pin them for full speed):
    the copies overlap the fold chunk by chunk (repops_fixed_order_mean_sgd_host).
    Asynchronous on `stream`: synchronise it before reading theta."""
    nC = len(grads)
    for t in list(grads) + [theta]:
        if t.is_cuda or t.dtype.itemsize != 4 or not t.is_contiguous() or t.numel() != theta.numel():
            raise ValueError("gradients and theta must be contiguous float32 CPU tensors of one size")
    if len(order) != nC:
        raise ValueError("order must have one entry per contributor")
    parr = (ctypes.c_void_p * max(nC, 1))(*[g.data_ptr() for g in grads])
    oarr = (ctypes.c_int * max(nC, 1))(*[int(x) for x in order])
    rc = load().repops_fixed_order_mean_sgd_host(nC, theta.numel(), ctypes.cast(parr, ctypes.c_void_p),
                                                 ctypes.cast(oarr, ctypes.c_void_p), ctypes.c_float(eta),
                                                 theta.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_fixed_order_mean_sgd_host")
    return theta


def merkle_sha256_host(t, leaf: int = 4096, out=None, *, stream=None):
    """Merkle root of a contiguous CPU tensor's bytes (pin it for full speed)
    into `out` (a 32-byte uint8 CPU tensor, allocated if None): chunks are
    copied in while the previous chunk is hashed (repops_merkle_sha256_host).
    Asynchronous on `stream`: synchronise it before reading out."""
    import torch
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("t must be a contiguous CPU tensor")
    if out is None:
        out = torch.zeros(32, dtype=torch.uint8, pin_memory=t.is_pinned())
    if out.is_cuda or out.dtype != torch.uint8 or out.numel() != 32:
        raise ValueError("out must be a 32-byte uint8 CPU tensor")
    rc = load().repops_merkle_sha256_host(t.data_ptr(), t.numel() * t.element_size(), leaf, out.data_ptr(),
                                          _stream_handle(stream))
    _capi.check(rc, "repops_merkle_sha256_host")
    return out


def merkle_workspace_bytes(nbytes: int, leaf: int = 4096) -> int:
    return load().repops_merkle_workspace_bytes(nbytes, leaf)


def merkle_sha256(t, leaf: int = 4096, out=None, *, nbytes: int = None, workspace=None,
                  stream=None):
    """32-byte SHA-256 Merkle root (uint8 CUDA tensor) of the bytes of `t`.

    t: a contiguous CUDA tensor; its storage bytes are hashed as stored.
    nbytes: hash only the first nbytes bytes.  workspace: optional uint8 CUDA
    tensor used as scratch; by default one comes from torch's caching
    allocator (the library's pool when `stream` is a raw handle)."""
    import torch
    L = load()
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("t must be a contiguous CUDA tensor")
    n = t.numel() * t.element_size() if nbytes is None else int(nbytes)
    if out is None:
        out = torch.empty(32, dtype=torch.uint8, device=t.device)
    s = _stream_handle(stream)
    if workspace is None:
        # the level scratch from torch's caching allocator where it can follow
        # the stream (repops_merkle_sha256_ws), else from the library's pool
        need = L.repops_merkle_workspace_bytes(n, leaf)
        workspace = _workspace(max(need, 16), t.device, stream) if need else None
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


def scratch_set_keep_bytes(nbytes: int) -> None:
    """Lets the library's scratch pool of the current device keep up to
    `nbytes` of freed scratch mapped across synchronisations (0, the default,
    keeps none; repops_scratch_set_keep_bytes)."""
    _capi.check(load().repops_scratch_set_keep_bytes(int(nbytes)), "repops_scratch_set_keep_bytes")


def scratch_release() -> None:
    """Hands the current device's unused scratch-pool memory back to the system
    (repops_scratch_release)."""
    _capi.check(load().repops_scratch_release(), "repops_scratch_release")


def scratch_reserved_bytes() -> int:
    """Device memory the library's scratch pool of the current device holds
    mapped (repops_scratch_reserved_bytes)."""
    v = ctypes.c_uint64(0)
    _capi.check(load().repops_scratch_reserved_bytes(ctypes.byref(v)), "repops_scratch_reserved_bytes")
    return v.value


class _HostBlock:
    """One repops_host_alloc allocation, exposed to NumPy (and through it to
    torch) by its array interface; unregistered and unmapped when the last
    array or tensor over it is gone."""

    def __init__(self, nbytes: int):
        p = ctypes.c_void_p()
        _capi.check(load().repops_host_alloc(int(nbytes), ctypes.byref(p)), "repops_host_alloc")
        self.ptr = p.value
        self.__array_interface__ = {"shape": (int(nbytes),), "typestr": "|u1", "data": (self.ptr, False),
                                    "version": 3}

    def __del__(self):
        if getattr(self, "ptr", None):
            try:
                load().repops_host_free(self.ptr)
            except Exception:   # interpreter shutdown: the process's memory goes anyway
                pass
            self.ptr = None


def host_empty(shape, dtype=None):
    """A contiguous CPU tensor over page-locked host memory in transparent huge
    pages (repops_host_alloc), for the host-buffer calls: zero-filled, freed
    when the tensor and every view of it are gone.  On a Grace host such
    buffers keep the copy engines at the link's rate where memory pinned in
    64 KB pages does not.

    Unlike PyTorch's pinned memory, nothing holds the block back for copies
    still in flight: keep a tensor (or a view of it) alive until every copy
    that reads or writes it has completed, e.g. until its stream is
    synchronised."""
    import numpy as np
    import torch
    dtype = torch.float32 if dtype is None else dtype
    shape = tuple(int(x) for x in shape) if isinstance(shape, (tuple, list)) else (int(shape),)
    if any(x < 0 for x in shape):
        raise ValueError("negative dimension in %s" % (shape,))
    n = 1
    for x in shape:
        n *= x
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    if nbytes == 0:
        return torch.empty(shape, dtype=dtype)
    if torch.cuda.is_available():
        torch.cuda.init()   # torch reports host memory as pinned only once its CUDA state exists
    return torch.from_numpy(np.asarray(_HostBlock(nbytes))).view(dtype).view(shape)


def set_thread_status_word(word=None) -> None:
    """Binds a caller-owned device status word (a 1-element int32/uint32 CUDA
    tensor, or None for the library's shared word) to this host thread's
    launches (see repops_set_thread_status_word)."""
    ptr = None
    if word is not None:
        if not word.is_cuda or word.element_size() != 4 or word.numel() < 1:
            raise ValueError("word must be a CUDA tensor of 4-byte elements")
        ptr = word.data_ptr()
    _capi.check(load().repops_set_thread_status_word(ptr), "repops_set_thread_status_word")


def merkle_tree(t, leaf: int = 4096, *, nbytes: int = None, tree=None, root=None, stream=None):
    """(tree, root): every node of the Merkle tree of t's bytes (uint8 CUDA
    tensor of shape (nodes, 32), leaf digests first, root last) and the root."""
    import torch
    L = load()
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("t must be a contiguous CUDA tensor")
    n = t.numel() * t.element_size() if nbytes is None else int(nbytes)
    need = L.repops_merkle_tree_bytes(n, leaf)
    if need == 0:
        raise ValueError("empty input or bad leaf size")
    if tree is None:
        tree = torch.empty((need // 32, 32), dtype=torch.uint8, device=t.device)
    if root is None:
        root = torch.empty(32, dtype=torch.uint8, device=t.device)
    rc = L.repops_merkle_tree_sha256(t.data_ptr(), n, leaf, tree.data_ptr(),
                                     tree.numel() * tree.element_size(), root.data_ptr(),
                                     _stream_handle(stream))
    _capi.check(rc, "repops_merkle_tree_sha256")
    return tree, root


def merkle_proof(tree, nleaves: int, index: int, *, stream=None):
    """(steps, 32) uint8 CUDA tensor: siblings of leaf `index`, bottom-up."""
    import torch
    L = load()
    steps = L.repops_merkle_proof_steps(nleaves, index)
    if steps < 0:
        raise RepopsError(steps, "repops_merkle_proof_steps")
    out = torch.empty((max(steps, 1), 32), dtype=torch.uint8, device=tree.device)
    rc = L.repops_merkle_proof(tree.data_ptr(), nleaves, index, out.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_merkle_proof")
    return out[:steps]


def merkle_verify(leaf_bytes, nleaves: int, index: int, proof, root, *, stream=None):
    """int32 CUDA tensor: 1 if leaf_bytes (a CUDA tensor's bytes) is leaf
    `index` of the tree with this root, else 0."""
    import torch
    L = load()
    ok = torch.empty(1, dtype=torch.int32, device=root.device)   # the kernel always writes it
    nb = leaf_bytes.numel() * leaf_bytes.element_size()
    rc = L.repops_merkle_verify(leaf_bytes.data_ptr() if nb else None, nb, nleaves, index,
                                proof.data_ptr() if proof.numel() else None, root.data_ptr(),
                                ok.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_merkle_verify")
    return ok


def replay(grads_per_step, orders, etas, theta, leaf: int = 4096, *, roots=None, stream=None):
    """Replays blocks in order: theta -= eta_t * mean_t (fixed order), then
    commits theta; returns the (steps, 32) uint8 CUDA tensor of roots."""
    import torch
    L = load()
    steps = len(grads_per_step)
    nC = len(grads_per_step[0]) if steps else 0
    flat_p, flat_o = [], []
    for gs, order in zip(grads_per_step, orders):
        if len(gs) != nC or len(order) != nC:
            raise ValueError("every block needs the same number of contributors")
        flat_p += [g if isinstance(g, int) else g.data_ptr() for g in gs]
        flat_o += [int(x) for x in order]
    parr = (ctypes.c_void_p * max(len(flat_p), 1))(*flat_p)
    oarr = (ctypes.c_int * max(len(flat_o), 1))(*flat_o)
    earr = (ctypes.c_float * max(steps, 1))(*[float(e) for e in etas])
    if roots is None:
        roots = torch.empty((steps, 32), dtype=torch.uint8, device=theta.device)
    rc = L.repops_replay_mean_sgd_commit(steps, nC, theta.numel(), ctypes.cast(parr, ctypes.c_void_p),
                                         ctypes.cast(oarr, ctypes.c_void_p), ctypes.cast(earr, ctypes.c_void_p),
                                         theta.data_ptr(), leaf, roots.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_replay_mean_sgd_commit")
    return roots


def _row_operand(x, name):
    import torch
    if x.dtype != torch.float32 or x.dim() != 2 or not x.is_cuda or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError("%s must be a 2-D float32 CUDA tensor with unit column stride" % name)
    return x.data_ptr(), max(x.stride(0), x.shape[1], 1)


def _row_out(x, out):
    import torch
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    if tuple(out.shape) != tuple(x.shape):
        raise ValueError("out must have the shape of x")
    return out


def attention_causal(q, k, v, out, *, seq_len: int, heads: int, kv_heads: int, scale: float, probs=None,
                     stream=None):
    """Fused causal grouped-query attention (repops_attention_causal_f32).

    q: (T, heads*dh), k and v: (T, kv_heads*dh), out: (T, heads*dh) float32
    CUDA views with unit column stride (any row pitch); T = sequences *
    seq_len.  probs: optional (sequences*heads, seq_len, seq_len) contiguous
    float32 tensor that receives every row of P.  Raises RepopsError
    (UNSUPPORTED) outside the kernel's limits."""
    L = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dim() != 2 or t.dtype.itemsize != 4 or (t.shape[1] > 1 and t.stride(1) != 1):
            raise ValueError("%s must be a 2-D float32 view with unit column stride" % name)
    T = q.shape[0]
    if T % seq_len:
        raise ValueError("rows are not a whole number of sequences")
    dh = q.shape[1] // heads
    pp = None
    if probs is not None:
        if not probs.is_contiguous() or probs.numel() != (T // seq_len) * heads * seq_len * seq_len:
            raise ValueError("probs must be a contiguous (sequences*heads, S, S) tensor")
        pp = probs.data_ptr()
    rc = L.repops_attention_causal_f32(T // seq_len, seq_len, heads, kv_heads, dh,
                                       q.data_ptr(), q.stride(0), k.data_ptr(), k.stride(0),
                                       v.data_ptr(), v.stride(0), float(scale), out.data_ptr(), out.stride(0),
                                       pp, _stream_handle(stream))
    _capi.check(rc, "repops_attention_causal_f32")
    return out


def softmax_rows(x, out=None, *, causal_first=None, causal_period=None, stream=None):
    """Row softmax with the order-fixed max/sum trees and the library's exp.
    causal_first=p: row i sees only its first p + (i mod causal_period) + 1
    values (queries at positions p, p + 1, ...; the period defaults to the row
    count), +0 after (repops_softmax_rows_causal_f32)."""
    L = load()
    px, ldx = _row_operand(x, "x")
    out = _row_out(x, out)
    py, ldy = _row_operand(out, "out")
    if causal_first is None:
        rc = L.repops_softmax_rows_f32(x.shape[0], x.shape[1], px, ldx, py, ldy, _stream_handle(stream))
        _capi.check(rc, "repops_softmax_rows_f32")
    else:
        period = int(causal_period) if causal_period is not None else max(x.shape[0], 1)
        rc = L.repops_softmax_rows_causal_f32(x.shape[0], x.shape[1], px, ldx, py, ldy, int(causal_first),
                                              period, _stream_handle(stream))
        _capi.check(rc, "repops_softmax_rows_causal_f32")
    return out


def layernorm_rows(x, gamma, beta, eps: float = 1e-5, out=None, *, stream=None):
    L = load()
    px, ldx = _row_operand(x, "x")
    out = _row_out(x, out)
    py, ldy = _row_operand(out, "out")
    if gamma.numel() != x.shape[1] or beta.numel() != x.shape[1]:
        raise ValueError("gamma and beta need one value per column")
    rc = L.repops_layernorm_rows_f32(x.shape[0], x.shape[1], px, ldx, gamma.data_ptr(), beta.data_ptr(),
                                     ctypes.c_float(eps), py, ldy, _stream_handle(stream))
    _capi.check(rc, "repops_layernorm_rows_f32")
    return out


def rmsnorm_rows(x, gamma, eps: float = 1e-6, out=None, *, stream=None):
    L = load()
    px, ldx = _row_operand(x, "x")
    out = _row_out(x, out)
    py, ldy = _row_operand(out, "out")
    if gamma.numel() != x.shape[1]:
        raise ValueError("gamma needs one value per column")
    rc = L.repops_rmsnorm_rows_f32(x.shape[0], x.shape[1], px, ldx, gamma.data_ptr(), ctypes.c_float(eps),
                                   py, ldy, _stream_handle(stream))
    _capi.check(rc, "repops_rmsnorm_rows_f32")
    return out


def gelu(x, out=None, *, stream=None):
    """Elementwise GeLU (erf form) of a contiguous float32 CUDA tensor."""
    import torch
    L = load()
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty_like(x)
    rc = L.repops_gelu_f32(x.numel(), x.data_ptr(), out.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_gelu_f32")
    return out


def convert(x, dtype, out=None, *, stream=None):
    """x converted to `dtype` (float32, float16, bfloat16): exact widening,
    round-to-nearest-even narrowing (repops_convert).  x: contiguous CUDA tensor."""
    import torch
    st, dt = _storage_type(x.dtype), _storage_type(dtype)
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty(x.shape, dtype=dtype, device=x.device)
    if out.dtype != dtype or out.numel() != x.numel() or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of dtype %s with x's size" % dtype)
    rc = load().repops_convert(x.numel(), x.data_ptr(), st, out.data_ptr(), dt, _stream_handle(stream))
    _capi.check(rc, "repops_convert")
    return out


def _typed_operand(X, name):
    """(pointer, leading dim, transposed) of a 2-D CUDA view of any storage type."""
    if X.dim() != 2 or not X.is_cuda:
        raise TypeError("%s must be a 2-D CUDA tensor" % name)
    r, c = X.shape
    s0, s1 = X.stride()
    if s1 == 1 and s0 >= max(c, 1):
        return X.data_ptr(), s0, 0
    if s0 == 1 and s1 >= max(r, 1):
        return X.data_ptr(), s1, 1
    raise ValueError("%s must be row-major or a transposed (column-major) view" % name)


def gemm_typed(A, B, out=None, *, out_dtype=None, config: int = -1, loader: int = LOADER_AUTO, stream=None):
    """C = A @ B on operands stored as float32, float16 or bfloat16: widened
    exactly, the order-fixed binary32 k-chain, narrowed once to out's dtype
    (repops_gemm_typed).  out_dtype defaults to float32."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    pa, lda, ta = _typed_operand(A, "A")
    pb, ldb, tb = _typed_operand(B, "B")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    if out.dim() != 2 or tuple(out.shape) != (M, N) or (N > 0 and out.stride(1) != 1):
        raise ValueError("out must be (M, N) with unit column stride")
    rc = load().repops_gemm_typed(config, loader, ta, tb, M, N, K, pa, _storage_type(A.dtype), lda, pb,
                                  _storage_type(B.dtype), ldb, out.data_ptr(), _storage_type(out.dtype),
                                  max(out.stride(0), N, 1), _stream_handle(stream))
    _capi.check(rc, "repops_gemm_typed")
    return out


def rolling_hash(words, window: int, out=None, *, stream=None):
    """(rows, width - window + 1) Rabin-Karp window hashes modulo 2^61 - 1 of
    a (rows, width) batch of uint32 words (an int32 or uint32 CUDA tensor, its
    bits read as uint32; unit column stride).  Returned as int64 (every hash
    is below 2^61)."""
    import torch
    if words.dim() != 2 or not words.is_cuda or words.element_size() != 4 or words.dtype.is_floating_point:
        raise TypeError("words must be a 2-D 32-bit integer CUDA tensor")
    rows, width = words.shape
    if width > 0 and words.stride(1) != 1:
        raise ValueError("words must have unit column stride")
    n = width - window + 1
    if out is None:
        out = torch.empty((rows, max(n, 0)), dtype=torch.int64, device=words.device)
    if out.dtype != torch.int64 or tuple(out.shape) != (rows, max(n, 0)) or (n > 0 and out.stride(1) != 1):
        raise ValueError("out must be an int64 (rows, width - window + 1) tensor with unit column stride")
    rc = load().repops_rolling_hash_u32(rows, width, words.data_ptr(), max(words.stride(0), width, 1), window,
                                        out.data_ptr(), max(out.stride(0), n, 1), _stream_handle(stream))
    _capi.check(rc, "repops_rolling_hash_u32")
    return out


def colsum(x, out=None, *, stream=None):
    """Column sums of a 2-D float32 CUDA tensor (unit column stride), each over
    the 32-ary tree in row order (repops_colsum_f32)."""
    import torch
    rows, cols = x.shape
    px, ldx = _row_operand(x, "x") if rows else (x.data_ptr(), max(cols, 1))
    if out is None:
        out = torch.empty(cols, dtype=torch.float32, device=x.device)
    rc = load().repops_colsum_f32(rows, cols, px, ldx, out.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_colsum_f32")
    return out


def gelu_backward(x, dy, out=None, *, stream=None):
    """dy * GeLU'(x) for contiguous float32 CUDA tensors of one size."""
    import torch
    for t, n in ((x, "x"), (dy, "dy")):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous float32 CUDA tensor" % n)
    if x.numel() != dy.numel():
        raise ValueError("x and dy differ in size")
    if out is None:
        out = torch.empty_like(x)
    rc = load().repops_gelu_backward_f32(x.numel(), x.data_ptr(), dy.data_ptr(), out.data_ptr(),
                                         _stream_handle(stream))
    _capi.check(rc, "repops_gelu_backward_f32")
    return out


def rmsnorm_backward(x, gamma, eps, dy, dx=None, dyxh=None, *, res=None, stream=None):
    """(dx, dy * xhat) of RMSNorm rows (repops_rmsnorm_backward_f32), dx + res
    when res is given (res may be dx); colsum(dy * xhat) is dgamma."""
    px, ldx = _row_operand(x, "x")
    pd, ldd = _row_operand(dy, "dy")
    dx = _row_out(x, dx)
    dyxh = _row_out(x, dyxh)
    pdx, lddx = _row_operand(dx, "dx")
    pp, ldp = _row_operand(dyxh, "dyxh")
    pr, ldr = _row_operand(res, "res") if res is not None else (None, 0)
    if gamma.numel() != x.shape[1] or tuple(dy.shape) != tuple(x.shape) or \
            (res is not None and tuple(res.shape) != tuple(x.shape)):
        raise ValueError("gamma needs one value per column; dy and res x's shape")
    rc = load().repops_rmsnorm_backward_f32(x.shape[0], x.shape[1], px, ldx, gamma.data_ptr(), ctypes.c_float(eps),
                                            pd, ldd, pr, ldr, pdx, lddx, pp, ldp, _stream_handle(stream))
    _capi.check(rc, "repops_rmsnorm_backward_f32")
    return dx, dyxh


def softmax_backward(p, dp, out=None, *, causal_first=None, causal_period=None, stream=None):
    """p * (dp - rowsum(dp * p)) (repops_softmax_backward_f32); out may be dp.
    causal_first / causal_period: the backward of softmax_rows with the same
    arguments -- row i covers its prefix only, +0 after, and never reads dp
    past it (repops_softmax_backward_causal_f32)."""
    pp, ldp = _row_operand(p, "p")
    pg, ldg = _row_operand(dp, "dp")
    out = _row_out(p, out)
    po, ldo = _row_operand(out, "out")
    if tuple(dp.shape) != tuple(p.shape):
        raise ValueError("p and dp differ in shape")
    if causal_first is None:
        rc = load().repops_softmax_backward_f32(p.shape[0], p.shape[1], pp, ldp, pg, ldg, po, ldo,
                                                _stream_handle(stream))
        _capi.check(rc, "repops_softmax_backward_f32")
    else:
        period = int(causal_period) if causal_period is not None else max(p.shape[0], 1)
        rc = load().repops_softmax_backward_causal_f32(p.shape[0], p.shape[1], pp, ldp, pg, ldg, po, ldo,
                                                       int(causal_first), period, _stream_handle(stream))
        _capi.check(rc, "repops_softmax_backward_causal_f32")
    return out


def swiglu(g, u, out=None, *, stream=None):
    """SiLU(g) * u element by element (repops_swiglu_f32); g, u and out are
    2-D float32 CUDA tensors of one shape with unit column stride (column
    blocks of a wider matrix are fine); out may be g or u."""
    pg, ldg = _row_operand(g, "g")
    pu, ldu = _row_operand(u, "u")
    out = _row_out(g, out)
    ph, ldh = _row_operand(out, "out")
    if tuple(u.shape) != tuple(g.shape):
        raise ValueError("g and u differ in shape")
    rc = load().repops_swiglu_f32(g.shape[0], g.shape[1], pg, ldg, pu, ldu, ph, ldh, _stream_handle(stream))
    _capi.check(rc, "repops_swiglu_f32")
    return out


def swiglu_backward(g, u, dh, dg=None, du=None, *, stream=None):
    """(dg, du) of h = SiLU(g) * u given dh (repops_swiglu_backward_f32); dg
    may be g or dh, du may be u or dh."""
    pg, ldg = _row_operand(g, "g")
    pu, ldu = _row_operand(u, "u")
    pd, ldd = _row_operand(dh, "dh")
    dg = _row_out(g, dg)
    du = _row_out(g, du)
    pdg, lddg = _row_operand(dg, "dg")
    pdu, lddu = _row_operand(du, "du")
    if tuple(u.shape) != tuple(g.shape) or tuple(dh.shape) != tuple(g.shape):
        raise ValueError("g, u and dh differ in shape")
    rc = load().repops_swiglu_backward_f32(g.shape[0], g.shape[1], pg, ldg, pu, ldu, pd, ldd, pdg, lddg, pdu, lddu,
                                           _stream_handle(stream))
    _capi.check(rc, "repops_swiglu_backward_f32")
    return dg, du


def rope_frequencies(pairs: int, ln_base: float, device="cuda", *, stream=None):
    """f_i = exp(-((i / pairs) * ln_base)), i < pairs, with ln_base rounded to
    binary32 (repops_rope_frequencies_f32)."""
    import torch
    out = torch.empty(pairs, dtype=torch.float32, device=device)
    rc = load().repops_rope_frequencies_f32(pairs, ctypes.c_float(ln_base), out.data_ptr(), _stream_handle(stream))
    _capi.check(rc, "repops_rope_frequencies_f32")
    return out


def rope_table(positions: int, freq, *, stream=None):
    """(cos, sin), each positions x pairs, of the angles p * freq[i]
    (repops_rope_table_f32)."""
    import torch
    if freq.dtype != torch.float32 or not freq.is_cuda or not freq.is_contiguous() or freq.dim() != 1:
        raise ValueError("freq must be a contiguous float32 CUDA vector")
    c = torch.empty(positions, freq.numel(), dtype=torch.float32, device=freq.device)
    s = torch.empty_like(c)
    rc = load().repops_rope_table_f32(positions, freq.numel(), freq.data_ptr(), c.data_ptr(), s.data_ptr(),
                                      _stream_handle(stream))
    _capi.check(rc, "repops_rope_table_f32")
    return c, s


def rope(x, heads: int, cos, sin, *, first: int = 0, period: int = None, inverse: bool = False, stream=None):
    """Rotates, in place, the adjacent pairs of the first `heads` heads of
    every row of x (2-D float32 CUDA, unit column stride; head width 2 *
    cos.shape[1]) to position first + (row mod period) (repops_rope_f32);
    inverse=True applies the transpose (the backward).  Returns x."""
    px, ldx = _row_operand(x, "x")
    for t, n in ((cos, "cos"), (sin, "sin")):
        if not t.is_contiguous() or t.dim() != 2 or t.shape != cos.shape:
            raise ValueError("%s must be a contiguous positions x pairs table" % n)
    positions, pairs = cos.shape
    per = int(period) if period is not None else max(x.shape[0], 1)
    rc = load().repops_rope_f32(x.shape[0], heads, pairs, px, ldx, cos.data_ptr(), sin.data_ptr(), positions,
                                int(first), per, int(bool(inverse)), _stream_handle(stream))
    _capi.check(rc, "repops_rope_f32")
    return x
