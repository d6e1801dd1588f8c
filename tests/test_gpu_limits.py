"""GPU parity at the size limits: outputs and buffers past 2^31 elements (and a
commitment past 2^32 bytes), where 32-bit index arithmetic would wrap.  The
oracle checks sampled rows or slices (elements and rows are independent, so
the oracle on a sample is exact) and the full Merkle root.

Each case holds 9-26 GB on the device; the bar is bit-exact.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda:0"
BIG = (1 << 31) + 5


def u32(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def sample(n, count, seed):
    g = torch.Generator().manual_seed(seed)
    picks = {0, 1, n - 1, n - 2} | {int(x) for x in torch.randint(0, n, (count,), generator=g)}
    return sorted(picks)


def test_gemm_output_past_2_31_elements(rp, orc):
    # C is 65539 x 32771 = 2,147,778,769 elements (8.6 GB); K = 8
    M, N, K = 65539, 32771, 8
    A = inputs.normal((M, K), 1.0, 900, DEV)
    B = inputs.normal((K, N), 1.0, 901, DEV)
    C = rp.gemm(A, B)
    rows = sample(M, 12, 902)
    want = orc.gemm(A[rows].cpu().numpy(), B.cpu().numpy())
    assert np.array_equal(u32(C[rows].cpu().numpy()), u32(want))
    del C
    # the transposed-A storage and the cp.async loader reach the same rows
    At = A.t().contiguous()
    C2 = rp.gemm(At.t(), B, loader=rp.LOADER_CPASYNC)
    assert np.array_equal(u32(C2[rows].cpu().numpy()), u32(want))


def test_batched_gemm_strides_past_2_31(rp, orc):
    # two 46341 x 46341 outputs (2,147,488,281 elements each) stacked, with an
    # in-place residual epilogue
    M = N = 46341
    K = 4
    A = inputs.normal((2, M, K), 1.0, 910, DEV)
    B = inputs.normal((2, K, N), 1.0, 911, DEV)
    C = inputs.normal((2, M, N), 1.0, 912, DEV)
    rows = sample(M, 6, 913)
    before = C[:, rows].cpu().numpy()
    rp.gemm_batched(A, B, out=C, alpha=0.5, residual=C)
    for b in range(2):
        prod = orc.gemm(A[b, rows].cpu().numpy(), B[b].cpu().numpy())
        want = ((prod * np.float32(0.5)).astype(np.float32) + before[b]).astype(np.float32)
        assert np.array_equal(u32(C[b, rows].cpu().numpy()), u32(want)), b


def test_mean_sgd_past_2_31_elements(rp, orc):
    # 2 contributors x (2^31 + 5) fp32 and theta: 26 GB
    grads = [inputs.normal((BIG,), 1e-2, 920 + r, DEV) for r in range(2)]
    theta = inputs.normal((BIG,), 0.02, 922, DEV)
    starts = [0, (1 << 31) - 2048, BIG - 4096] + sample(BIG - 4096, 5, 923)
    before = {s: theta[s:s + 4096].cpu().numpy() for s in starts}
    rp.fixed_order_mean_sgd(grads, [1, 0], 1e-3, theta)
    torch.cuda.synchronize()
    for s in starts:
        want = orc.mean_sgd([g[s:s + 4096].cpu().numpy() for g in grads], [1, 0], 1e-3, before[s])
        assert np.array_equal(u32(theta[s:s + 4096].cpu().numpy()), u32(want)), s


def test_row_operators_past_2_31_elements(rp, orc):
    # 1,048,577 rows x 2052 values (2,151,680,004 elements): softmax, RMSNorm
    rows, cols = (1 << 20) + 1, 2052
    X = inputs.normal((rows, cols), 2.0, 930, DEV)
    g = inputs.normal((cols,), 1.0, 931, DEV)
    picks = sample(rows, 10, 932)
    Xs = X[picks].cpu().numpy()
    Y = rp.softmax_rows(X)
    assert np.array_equal(u32(Y[picks].cpu().numpy()), u32(orc.softmax_rows(Xs)))
    rp.rmsnorm_rows(X, g, 1e-5, out=Y)
    assert np.array_equal(u32(Y[picks].cpu().numpy()), u32(orc.rmsnorm_rows(Xs, g.cpu().numpy(), 1e-5)))


def test_merkle_past_2_32_bytes(rp, orc):
    # 4 GiB + 3 leaves + 100 bytes: byte offsets past 32 bits, a short last leaf
    n = (1 << 32) + 3 * 4096 + 100
    t = torch.randint(0, 256, (n,), dtype=torch.uint8, device=DEV,
                      generator=torch.Generator(device=DEV).manual_seed(940))
    got = bytes(rp.merkle_sha256(t).cpu().numpy())
    assert got == orc.merkle_root(t.cpu().numpy(), 4096)
