"""The host allocator behind the host-buffer calls (repops_host_alloc /
repops_host_free, the binding's host_empty): page-locked, zero-filled memory
at a huge-page-aligned address, released with its last tensor, and the
host-buffer GEMM, mean + SGD and Merkle root computed from it equal to the
device calls and the oracle.  A deployment aid; the pages have no counterpart.
"""
import ctypes
import gc
import os

import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def huge_page_bytes():
    """The transparent huge page size, or None where huge pages are off."""
    try:
        with open("/sys/kernel/mm/transparent_hugepage/enabled") as f:
            if "[never]" in f.read():
                return None
    except OSError:
        return None
    try:
        with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
            return int(f.read())
    except (OSError, ValueError):
        return 2 << 20


def test_host_empty_is_pinned_zero_and_aligned(rp):
    for shape, dtype in (((1000,), torch.float32), ((3, 5), torch.uint8), ((7, 9), torch.float16)):
        t = rp.host_empty(shape, dtype)
        assert tuple(t.shape) == shape and t.dtype == dtype and t.is_contiguous()
        assert t.is_pinned() and not t.is_cuda
        assert t.data_ptr() % os.sysconf("SC_PAGE_SIZE") == 0
        assert int(t.view(torch.uint8).sum()) == 0
        t.fill_(7)
        assert torch.equal(t, torch.full(shape, 7, dtype=dtype))
    # at least one huge page: its start is aligned to the huge page size
    hp = huge_page_bytes()
    if hp is None:
        return   # huge pages off: ordinary pages, nothing more to check
    big = rp.host_empty((hp // 4 + 1000,), torch.float32)
    assert big.data_ptr() % hp == 0
    big[-1] = 3.0
    assert float(big[-1]) == 3.0 and float(big[0]) == 0.0
    # a quarter of a huge page or more: rounded up to whole huge pages, so
    # its start is aligned to one too
    mid = rp.host_empty((hp // 4,), torch.uint8)
    assert mid.data_ptr() % hp == 0 and mid.numel() == hp // 4
    mid[-1] = 9
    assert int(mid[-1]) == 9 and int(mid[0]) == 0
    # empty shapes need no memory
    assert rp.host_empty((0, 4)).numel() == 0


def test_host_memory_lives_as_long_as_a_view(rp):
    t = rp.host_empty((4096,), torch.float32)
    t.copy_(torch.arange(4096, dtype=torch.float32))
    v = t[100:200]
    ptr = t.data_ptr()
    del t
    gc.collect()
    assert torch.equal(v, torch.arange(100, 200, dtype=torch.float32))
    d = v.to(DEV, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(d.cpu(), torch.arange(100, 200, dtype=torch.float32))
    del v, d
    gc.collect()
    # the block is gone: freeing its address again is refused
    assert rp.load().repops_host_free(ptr) == -1


def test_host_alloc_and_free_through_the_c_abi(rp):
    L = rp.load()
    p = ctypes.c_void_p()
    assert L.repops_host_alloc(3 * (1 << 20) + 17, ctypes.byref(p)) == 0 and p.value
    buf = (ctypes.c_uint8 * 64).from_address(p.value)
    buf[:] = bytes(range(64))
    assert bytes(buf) == bytes(range(64))
    assert L.repops_host_free(p.value) == 0
    assert L.repops_host_free(p.value) == -1          # already freed


def test_host_buffer_calls_from_the_allocator_match(rp, orc):
    # the three host-buffer calls on host_empty buffers give the device calls'
    # bits and the oracle's root
    M, N, K = 300, 200, 777
    A = inputs.normal((M, K), 1.0, 61, DEV)
    B = inputs.normal((K, N), 1.0, 62, DEV)
    hA, hB = rp.host_empty((M, K)), rp.host_empty((K, N))
    hA.copy_(A)
    hB.copy_(B)
    hC = rp.host_empty((M, N))
    s = torch.cuda.current_stream()
    rp.gemm_host(hA, hB, out=hC, stream=s)
    C = rp.gemm(A, B)
    s.synchronize()
    assert torch.equal(hC.view(torch.int32), C.cpu().view(torch.int32))
    n, nC = 100_003, 5
    grads = [inputs.normal((n,), 1e-2, 63 + r, DEV) for r in range(nC)]
    theta = inputs.normal((n,), 0.02, 70, DEV)
    hg = [rp.host_empty((n,)) for _ in range(nC)]
    for h, g in zip(hg, grads):
        h.copy_(g)
    ht = rp.host_empty((n,))
    ht.copy_(theta)
    order = [3, 0, 4, 1, 2]
    rp.fixed_order_mean_sgd_host(hg, order, 1e-3, ht, stream=s)
    rp.fixed_order_mean_sgd(grads, order, 1e-3, theta)
    torch.cuda.synchronize()
    assert torch.equal(ht.view(torch.int32), theta.cpu().view(torch.int32))
    root = rp.host_empty((32,), torch.uint8)
    rp.merkle_sha256_host(hC, 4096, out=root, stream=s)
    s.synchronize()
    assert bytes(root.numpy()) == orc.merkle_root(hC.numpy(), 4096)
