"""Seeded random parity cases for the fixed-order mean + SGD ("Zoo Per-LLM
Chain Soundness" §2 "Aggregation rule", §5 "Determinism of left-fold",
"Update step") and the SHA-256 Merkle commitment (§1, §6, §7; "Verde与RepOps"
§2.3.2), through every entry point that computes them.

Mean + SGD: 1 to 64 contributors (a few cases up to 1024), 1 to 300,000
elements, float32, binary16 or bfloat16 gradients, each gradient and theta at
a random element offset (so most are not 16-byte aligned), a random fold
order and step size, on the device or from host buffers.  Merkle: 1 byte to
6 MiB at a random byte offset, leaves of 64 bytes to 64 KiB, through the
allocating call (pool scratch), a caller workspace, the binding (a workspace
from torch's caching allocator), the allocation-free call, the stored tree
and the host-buffer call.  Every theta element and every root byte must equal
the oracle's.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
F32, F16, BF16 = 0, 1, 2
TORCH = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}


def host_storage(t):
    """The oracle's view of a tensor: float32 values or the uint16 half bits."""
    if t.dtype == torch.float32:
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("case", range(120))
def test_random_mean_sgd_case_matches_oracle(rp, orc, case):
    rng = np.random.default_rng(7_000 + case)
    nC = int(rng.integers(1, 65)) if case % 10 else int(rng.integers(65, 1025))
    n = int(np.exp(rng.uniform(0.0, np.log(300_000.0)))) if case % 10 else int(rng.integers(1, 5_000))
    gtype = [F32, F16, BF16][int(rng.integers(3))]
    host = gtype == F32 and rng.integers(4) == 0
    eta = float(np.float32(rng.choice([-1.0, 1.0]) * 10.0 ** rng.uniform(-4, 0)))
    order = [int(x) for x in rng.permutation(nC)]
    grads = []
    for r in range(nC):
        off = int(rng.integers(0, 4))
        g = inputs.normal((n + off,), 10.0 ** rng.uniform(-3, 1), 7_100 + 1031 * case + r, DEV)
        grads.append(g[off:off + n].to(TORCH[gtype]))
    off = int(rng.integers(0, 4))
    theta_buf = inputs.normal((n + off + 2,), 0.02, 7_099 + case, DEV)
    theta = theta_buf[off:off + n]
    want = orc.mean_sgd_typed([host_storage(g) for g in grads], gtype, order, eta, theta.cpu().numpy())
    before = theta_buf.clone()
    if host:
        hg = [g.cpu() for g in grads]
        ht = theta.cpu()
        s = torch.cuda.current_stream()
        rp.fixed_order_mean_sgd_host(hg, order, eta, ht, stream=s)
        s.synchronize()
        got = ht.numpy()
    else:
        rp.fixed_order_mean_sgd(grads, order, eta, theta)
        torch.cuda.synchronize()
        got = theta.cpu().numpy()
        # the elements around theta are untouched
        assert torch.equal(theta_buf[:off], before[:off]) and torch.equal(theta_buf[off + n:], before[off + n:])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan), (case, nC, n, gtype, host)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32)), (case, nC, n, gtype, host)


@pytest.mark.parametrize("case", range(120))
def test_random_merkle_case_matches_oracle(rp, orc, case):
    rng = np.random.default_rng(9_000 + case)
    nbytes = int(np.exp(rng.uniform(0.0, np.log(6 << 20))))
    leaf = 64 * int(np.exp(rng.uniform(0.0, np.log(1024.0))))
    off = int(rng.integers(0, 16))
    g = torch.Generator(device=DEV).manual_seed(9_000 + case)
    buf = torch.randint(0, 256, (off + nbytes + 16,), generator=g, dtype=torch.uint8, device=DEV)
    data = buf[off:off + nbytes]
    want = orc.merkle_root(data.cpu().numpy(), leaf)
    path = ["device", "workspace", "noalloc", "tree", "host", "binding"][case % 6]
    if path == "device":
        # the C entry point itself: scratch from the library's pool
        root = torch.empty(32, dtype=torch.uint8, device=DEV)
        rc = rp.load().repops_merkle_sha256(data.data_ptr(), nbytes, leaf, root.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
        assert rc == 0, rc
    elif path == "binding":
        root = rp.merkle_sha256(data, leaf)
    elif path == "workspace":
        need = rp.merkle_workspace_bytes(nbytes, leaf)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=DEV)
        root = rp.merkle_sha256(data, leaf, workspace=ws)
    elif path == "noalloc":
        root = torch.empty(32, dtype=torch.uint8, device=DEV)
        L = rp.load()
        rc = L.repops_merkle_sha256_noalloc(data.data_ptr(), nbytes, leaf, root.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
        assert rc == 0, rc
    elif path == "tree":
        tree, root = rp.merkle_tree(data, leaf)
        torch.cuda.synchronize()
        assert np.array_equal(tree.cpu().numpy(), orc.merkle_tree(data.cpu().numpy(), leaf)), (case, nbytes, leaf)
    else:
        hb = data.cpu()
        s = torch.cuda.current_stream()
        root = rp.merkle_sha256_host(hb, leaf, stream=s)
        s.synchronize()
    torch.cuda.synchronize()
    assert bytes(root.cpu().numpy()) == want, (case, nbytes, leaf, off, path)
