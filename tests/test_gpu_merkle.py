"""GPU parity of the SHA-256 Merkle commitment against the oracle.

"Zoo Per-LLM Chain Soundness" §1, §6, §7; "Verde与RepOps" §2.3.2.  Bar:
byte-identical roots.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def dev_bytes(n, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randint(0, 256, (n,), generator=g, device=DEV, dtype=torch.uint8)


def root(rp, t, leaf=4096, **kw):
    r = rp.merkle_sha256(t, leaf, **kw)
    torch.cuda.synchronize()
    return r.cpu().numpy().tobytes()


@pytest.mark.parametrize("n", [1, 63, 64, 65, 4095, 4096, 4097, 8192, 3 * 4096 + 5,
                               128 * 4096, 128 * 4096 + 1, 129 * 4096 + 100, 1000 * 4096,
                               300 * 128 * 4096 + 17])
def test_merkle_roots_match_oracle(rp, orc, n):
    t = dev_bytes(n, n % 1000)
    assert root(rp, t) == orc.merkle_root(t.cpu().numpy(), 4096)


@pytest.mark.parametrize("leaf", [64, 128, 1024, 65536])
def test_merkle_other_leaf_sizes(rp, orc, leaf):
    for n in (leaf, 5 * leaf + 3, 300 * leaf):
        t = dev_bytes(n, leaf + n)
        assert root(rp, t, leaf) == orc.merkle_root(t.cpu().numpy(), leaf), (leaf, n)


def test_merkle_unaligned_input_and_workspace(rp, orc):
    n = 777 * 4096 + 123
    buf = dev_bytes(n + 16, 5)
    t = buf[3:3 + n]          # not 16-byte aligned: generic leaf path
    want = orc.merkle_root(t.cpu().numpy(), 4096)
    assert root(rp, t) == want
    ws = torch.empty(rp.merkle_workspace_bytes(n, 4096), dtype=torch.uint8, device=DEV)
    assert root(rp, t, workspace=ws) == want
    aligned = t.clone()
    assert root(rp, aligned) == want


def test_merkle_float_tensor_bytes_little_endian(rp, orc):
    x = inputs.normal((1 << 20,), 0.02, 300, DEV)
    assert root(rp, x) == orc.merkle_root(x.cpu().numpy(), 4096)


def test_merkle_detects_one_bit_flip(rp):
    x = inputs.normal((1 << 20,), 0.02, 301, DEV)
    r0 = root(rp, x)
    y = x.clone()
    y.view(torch.int32)[123457] ^= 1
    assert root(rp, y) != r0


@pytest.mark.slow
def test_merkle_1gib_tensor(rp, orc):
    # 2^28 fp32 (1 GiB), N(0, 0.02): 2^18 leaves, 2048 leaf CTAs (a full GPU)
    x = inputs.normal((1 << 28,), 0.02, 302, DEV)
    assert root(rp, x) == orc.merkle_root(x.cpu().numpy(), 4096)


@pytest.mark.slow
def test_merkle_4gib_tensor(rp, orc):
    # 2^30 fp32 (4 GiB), N(0, 0.02), 4096-byte leaves: 2^20 leaves
    x = inputs.normal((inputs.MERKLE_ELEMS,), 0.02, 300, DEV)
    got = root(rp, x)
    assert got == orc.merkle_root(x.cpu().numpy(), 4096)


def test_sha256_rate_probe_digests(rp):
    # thread t hashes its 64-byte block (big-endian words 16t .. 16t + 15)
    # repeated `iters` times; hashlib is the reference
    import hashlib
    import struct
    for iters in (0, 1, 3):
        D = rp.sha256_rate_probe(256, iters)
        torch.cuda.synchronize()
        got = D.cpu().numpy().astype(np.uint32)
        for t in (0, 1, 127, 255):
            block = struct.pack(">16I", *[16 * t + i for i in range(16)])
            want = hashlib.sha256(block * iters).digest()
            assert struct.pack(">8I", *got[t]) == want, (iters, t)
    with pytest.raises(rp.RepopsError):
        rp.sha256_rate_probe(100, 1)


@pytest.mark.parametrize("nbytes,leaf,pinned", [(700 * 128 * 4096 + 333, 4096, True), (77 * 4096 + 5, 4096, False),
                                                (300 * 1024 * 1024 + 64, 64, True), (1, 4096, True)])
def test_host_buffer_merkle_same_root(rp, orc, nbytes, leaf, pinned):
    # chunked copies of whole 128-leaf groups, the leaf kernel per chunk, the
    # upper levels once: the root equals the device call's and the oracle's
    g = torch.Generator().manual_seed(nbytes % 1000)
    t = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8)
    if pinned:
        t = t.pin_memory()
    s = torch.cuda.Stream()
    root = rp.merkle_sha256_host(t, leaf, stream=s)
    s.synchronize()
    assert bytes(root.numpy()) == rp.merkle_sha256(t.to(DEV), leaf).cpu().numpy().tobytes()
    if nbytes < (1 << 30):
        assert bytes(root.numpy()) == orc.merkle_root(t.numpy(), leaf)
