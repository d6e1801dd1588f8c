"""GPU parity of the backward operators of a training step (column sums, GeLU,
RMSNorm and softmax backward) against the oracle, through the C ABI.

"Verde与RepOps" §3.2, §4.3.  Bar: bit-exact, over single and multi-level
column trees, aligned, unaligned and in-place element-wise calls, and rows
from one value to several tree levels.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def u32(a):
    return np.ascontiguousarray(a).view(np.uint32)


@pytest.mark.parametrize("rows,cols,pad", [(1, 7, 0), (31, 100, 0), (32, 33, 3), (33, 64, 0), (1025, 300, 1),
                                           (40000, 17, 0), (4096, 2048, 0)])
def test_colsum_matches_oracle(rp, orc, rows, cols, pad):
    x = inputs.normal((rows, cols + pad), 1.0, rows + cols, DEV)[:, :cols]
    y = rp.colsum(x)
    assert np.array_equal(u32(y.cpu().numpy()), u32(orc.colsum(x.cpu().numpy())))


def test_colsum_of_no_rows_is_zero(rp):
    y = rp.colsum(torch.empty(0, 5, device=DEV))
    assert torch.equal(y, torch.zeros(5, device=DEV)) and not torch.signbit(y).any()


@pytest.mark.parametrize("n", [1, 7, 4096, (1 << 20) + 3])
def test_gelu_backward_matches_oracle(rp, orc, n):
    x = inputs.normal((n,), 3.0, 100 + n, DEV)
    dy = inputs.normal((n,), 1.0, 200 + n, DEV)
    want = orc.gelu_backward(x.cpu().numpy(), dy.cpu().numpy())
    assert np.array_equal(u32(rp.gelu_backward(x, dy).cpu().numpy()), u32(want))
    base = inputs.normal((n + 1,), 3.0, 300 + n, DEV)
    xs = base[1:]                                         # 4-byte aligned only
    assert np.array_equal(u32(rp.gelu_backward(xs, dy).cpu().numpy()),
                          u32(orc.gelu_backward(xs.cpu().numpy(), dy.cpu().numpy())))
    d2 = dy.clone()
    rp.gelu_backward(x, d2, out=d2)                       # in place over dy
    assert np.array_equal(u32(d2.cpu().numpy()), u32(want))


@pytest.mark.parametrize("rows,cols", [(5, 1), (5, 33), (7, 100), (64, 2048), (33, 4092), (9, 8192), (3, 8193),
                                       (2, 40000)])
def test_rmsnorm_backward_matches_oracle(rp, orc, rows, cols):
    x = inputs.normal((rows, cols), 1.0, 400 + cols, DEV)
    g = inputs.normal((cols,), 1.0, 401, DEV)
    dy = inputs.normal((rows, cols), 1.0, 402 + cols, DEV)
    dx, p = rp.rmsnorm_backward(x, g, 1e-5, dy)
    wdx, wp = orc.rmsnorm_backward(x.cpu().numpy(), g.cpu().numpy(), 1e-5, dy.cpu().numpy())
    assert np.array_equal(u32(dx.cpu().numpy()), u32(wdx))
    assert np.array_equal(u32(p.cpu().numpy()), u32(wp))
    assert np.array_equal(u32(rp.colsum(p).cpu().numpy()), u32(orc.colsum(wp)))
    res = inputs.normal((rows, cols), 1.0, 403 + cols, DEV)
    wdx2, _ = orc.rmsnorm_backward(x.cpu().numpy(), g.cpu().numpy(), 1e-5, dy.cpu().numpy(), res.cpu().numpy())
    d2 = res.clone()
    rp.rmsnorm_backward(x, g, 1e-5, dy, dx=d2, res=d2)                  # residual added in place
    assert np.array_equal(u32(d2.cpu().numpy()), u32(wdx2))


@pytest.mark.parametrize("rows,cols", [(4, 1), (6, 33), (256, 2048), (3, 40000)])
def test_softmax_backward_matches_oracle(rp, orc, rows, cols):
    s = inputs.normal((rows, cols), 2.0, 500 + cols, DEV)
    p = rp.softmax_rows(s)
    dp = inputs.normal((rows, cols), 1.0, 501 + cols, DEV)
    want = orc.softmax_backward(p.cpu().numpy(), dp.cpu().numpy())
    assert np.array_equal(u32(rp.softmax_backward(p, dp).cpu().numpy()), u32(want))
    d2 = dp.clone()
    rp.softmax_backward(p, d2, out=d2)                    # in place over dp
    assert np.array_equal(u32(d2.cpu().numpy()), u32(want))


def test_softmax_backward_of_a_causal_block(rp, orc):
    s = inputs.normal((3 * 128, 128), 2.0, 600, DEV)
    p = rp.softmax_rows(s, causal_first=0, causal_period=128)
    dp = inputs.normal((3 * 128, 128), 1.0, 601, DEV)
    ds = rp.softmax_backward(p, dp)
    want = orc.softmax_backward(orc.softmax_rows_causal(s.cpu().numpy(), 0, 128), dp.cpu().numpy())
    assert np.array_equal(u32(ds.cpu().numpy()), u32(want))
