"""The binding's host_empty over a stand-in allocator (no GPU): one
repops_host_alloc per tensor, the memory handed back by exactly one
repops_host_free once the tensor and every view of it are gone, nothing
allocated for empty shapes, and an allocator error raised without a free."""
import ctypes
import gc

import pytest
import torch

import verifiable_repops_gemm_gb300 as rp
from verifiable_repops_gemm_gb300 import _capi


class FakeLib:
    """repops_host_alloc / repops_host_free over ctypes buffers."""

    def __init__(self, fail=False):
        self.live = {}
        self.allocs = 0
        self.frees = []
        self.fail = fail

    def repops_host_alloc(self, nbytes, out):
        if self.fail:
            return _capi.ERR_CUDA
        buf = ctypes.create_string_buffer(int(nbytes))
        addr = ctypes.addressof(buf)
        self.live[addr] = buf
        self.allocs += 1
        ctypes.cast(out, ctypes.POINTER(ctypes.c_void_p))[0] = addr
        return 0

    def repops_host_free(self, ptr):
        self.frees.append(ptr)
        return 0 if self.live.pop(ptr, None) is not None else _capi.ERR_INVALID_ARG

    def repops_status_string(self, code):
        return b"stand-in"

    def repops_last_cuda_error(self):
        return 0


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    monkeypatch.setattr(rp, "load", lambda *a, **k: lib)
    monkeypatch.setattr(_capi, "load", lambda *a, **k: lib)
    monkeypatch.setattr(torch.cuda, "is_available", lambda: False)
    return lib


def test_one_allocation_freed_once_with_its_last_view(fake):
    t = rp.host_empty((3, 5), torch.float32)
    assert fake.allocs == 1 and tuple(t.shape) == (3, 5) and t.dtype == torch.float32
    t.copy_(torch.arange(15, dtype=torch.float32).view(3, 5))
    v = t[1]
    ptr = t.data_ptr()
    del t
    gc.collect()
    assert fake.frees == [] and torch.equal(v, torch.arange(5, 10, dtype=torch.float32))
    del v
    gc.collect()
    assert fake.frees == [ptr] and not fake.live


def test_dtypes_and_empty_shapes(fake):
    for dtype in (torch.uint8, torch.float16, torch.bfloat16, torch.int64):
        t = rp.host_empty((7,), dtype)
        assert t.dtype == dtype and t.numel() == 7 and t.is_contiguous()
        del t
    gc.collect()
    assert fake.allocs == 4 and len(fake.frees) == 4 and not fake.live
    e = rp.host_empty((0, 9))
    assert e.shape == (0, 9) and fake.allocs == 4        # nothing to allocate
    with pytest.raises(ValueError):
        rp.host_empty((-1, 2))


def test_allocator_error_raises_and_frees_nothing(monkeypatch):
    lib = FakeLib(fail=True)
    monkeypatch.setattr(rp, "load", lambda *a, **k: lib)
    monkeypatch.setattr(_capi, "load", lambda *a, **k: lib)
    monkeypatch.setattr(torch.cuda, "is_available", lambda: False)
    with pytest.raises(_capi.RepopsError):
        rp.host_empty((16,))
    gc.collect()
    assert lib.frees == []
