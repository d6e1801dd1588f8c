"""The allocation-free Merkle entry point, checked against the allocating one
and against the oracle's root of the same bytes.

repops_merkle_sha256_noalloc serves callers that cannot allocate device
memory when they hash (a framework that owns all device memory in its own
pool, a latency-critical path, a plug-in host that forbids allocations after
start-up).  Its scratch is a fixed 1 MiB array inside the library, shared by
every call.  These tests call it through the C ABI and require the same root
bytes as repops_merkle_sha256, and as the oracle's Merkle root of the
input's bytes, on two calls in a row, so that whatever the first call leaves
in the shared array cannot leak into the second.

This file is named to be collected last.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
LEAF = 4096


def _bytes(n, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randint(0, 256, (n,), generator=g, device=DEV, dtype=torch.uint8)


def _roots(L, t, n, stream):
    ref = torch.zeros(32, dtype=torch.uint8, device=DEV)
    got = torch.full((32,), 0xAA, dtype=torch.uint8, device=DEV)
    assert L.repops_merkle_sha256(t.data_ptr(), n, LEAF, ref.data_ptr(), stream) == 0
    assert L.repops_merkle_sha256_noalloc(t.data_ptr(), n, LEAF, got.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    return ref.cpu().numpy().tobytes(), got.cpu().numpy().tobytes()


def test_noalloc_matches_allocating_root_on_two_calls_in_a_row(rp, orc):
    L = rp.load()
    stream = torch.cuda.current_stream().cuda_stream
    # first a larger input (two reduce passes over the shared scratch), then a
    # smaller one with a ragged last leaf, so the second call runs over what the
    # first one left behind
    n1 = 700 * 128 * LEAF + 333
    n2 = 1000 * LEAF + 17
    t1, t2 = _bytes(n1, 1), _bytes(n2, 2)
    ref1, got1 = _roots(L, t1, n1, stream)
    ref2, got2 = _roots(L, t2, n2, stream)
    assert got1 == ref1
    assert got2 == ref2
    assert ref1 != ref2
    # the oracle's root of the same bytes (leaf SHA256(0x00 || bytes), node
    # SHA256(0x01 || left || right), an unpaired node promoted)
    assert got1 == orc.merkle_root(t1.cpu().numpy(), LEAF)
    assert got2 == orc.merkle_root(t2.cpu().numpy(), LEAF)


def test_noalloc_small_input_and_limit(rp, orc):
    L = rp.load()
    stream = torch.cuda.current_stream().cuda_stream
    # at most 128 leaves: no scratch needed
    n = 77 * LEAF + 5
    t = _bytes(n, 3)
    ref, got = _roots(L, t, n, stream)
    assert got == ref
    assert got == orc.merkle_root(t.cpu().numpy(), LEAF)
    # one CTA's worth of leaves (128) past the largest input the 1 MiB scratch
    # can serve is refused before anything runs (the pointer is never read)
    limit_leaves = 32704 * 128
    assert L.repops_merkle_workspace_bytes(limit_leaves * LEAF, LEAF) <= 1 << 20
    assert L.repops_merkle_workspace_bytes((limit_leaves + 128) * LEAF, LEAF) > 1 << 20
    out = torch.zeros(32, dtype=torch.uint8, device=DEV)
    too_big = (limit_leaves + 128) * LEAF
    fake = out.data_ptr() + (1 << 20)     # a span that cannot overlap `out`
    assert L.repops_merkle_sha256_noalloc(fake, too_big, LEAF, out.data_ptr(), stream) == -7
