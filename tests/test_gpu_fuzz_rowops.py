"""Seeded random parity cases for the order-fixed row operators ("Verde与RepOps"
§3.2: a fixed order for the order-critical dimensions; §4.3: the operators
behind the measured models' overhead): softmax, causal softmax, LayerNorm,
RMSNorm and GeLU.

Each case draws a shape (1 to 300 rows, log-uniform; 1 to 40,000 columns,
log-uniform in even cases, uniform from 1,024 in odd ones),
an input view with a padded leading dimension and a random element offset
(so many rows are not 16-byte aligned and take the kernels' unaligned paths),
a value scale, and an output that is either the input itself (in place) or a
separately padded view between canary rows; causal cases draw `first` and the
period.  The row operators choose among several kernels by row length and
alignment (register-resident, staged, one warp per row, re-reading); every
output must equal the oracle's bit for bit (NaN where it is NaN) and the
canaries must survive.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CANARY = -3.5


def view(rng, rows, cols, seed, scale):
    pad = int(rng.integers(0, 8))
    off = int(rng.integers(0, 4))
    ld = cols + pad
    base = inputs.normal((off + (rows + 2) * ld,), scale, seed, DEV)
    return base, base[off + ld:off + ld + rows * ld].view(rows, ld)[:, :cols], off, ld


@pytest.mark.parametrize("case", range(400))
def test_random_row_operator_case_matches_oracle(rp, orc, case):
    rng = np.random.default_rng(11_000 + case)
    op = ["softmax", "causal", "layernorm", "rmsnorm", "gelu"][case % 5]
    rows = int(np.exp(rng.uniform(0.0, np.log(300.0))))
    if case % 2:
        cols = int(rng.integers(1024, 40_001))
    else:
        cols = int(np.exp(rng.uniform(0.0, np.log(40_000.0))))
    rows = max(1, min(rows, (4 << 20) // cols))
    scale = float(rng.choice([0.1, 1.0, 10.0]))
    if op == "gelu":
        x = inputs.normal((rows * cols,), scale, 11_500 + case, DEV)
        want = orc.gelu(x.cpu().numpy())
        got = rp.gelu(x) if case % 2 else rp.gelu(x, out=x)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32)), (case, rows * cols)
        return
    xbase, x, off, ld = view(rng, rows, cols, 11_100 + case, scale)
    xh = x.contiguous().cpu().numpy()
    in_place = bool(rng.integers(2))
    if in_place:
        out, ybase = x, xbase
    else:
        ypad, yoff = int(rng.integers(0, 8)), int(rng.integers(0, 4))
        ybase = torch.full((yoff + (rows + 2) * (cols + ypad),), CANARY, device=DEV)
        out = ybase[yoff + cols + ypad:yoff + (cols + ypad) * (rows + 1)].view(rows, cols + ypad)[:, :cols]
    what = dict(op=op, rows=rows, cols=cols, ld=ld, off=off, in_place=in_place)
    if op == "softmax":
        want = orc.softmax_rows(xh)
        rp.softmax_rows(x, out=out)
    elif op == "causal":
        first = int(rng.integers(0, cols))
        period = int(rng.integers(1, rows + 1))
        what.update(first=first, period=period)
        want = orc.softmax_rows_causal(xh, first, period)
        rp.softmax_rows(x, out=out, causal_first=first, causal_period=period)
    elif op == "layernorm":
        gamma = inputs.normal((cols,), 1.0, 11_200 + case, DEV)
        beta = inputs.normal((cols,), 0.1, 11_300 + case, DEV)
        want = orc.layernorm_rows(xh, gamma.cpu().numpy(), beta.cpu().numpy(), 1e-5)
        rp.layernorm_rows(x, gamma, beta, 1e-5, out=out)
    else:
        gamma = inputs.normal((cols,), 1.0, 11_400 + case, DEV)
        want = orc.rmsnorm_rows(xh, gamma.cpu().numpy(), 1e-6)
        rp.rmsnorm_rows(x, gamma, 1e-6, out=out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan), what
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32)), what
    if not in_place:
        # the rows above and below, and the padding of every row, untouched
        stride = out.stride(0)
        full = ybase[yoff:yoff + (rows + 2) * stride].view(rows + 2, stride)
        assert (full[0] == CANARY).all() and (full[rows + 1] == CANARY).all(), what
        assert (full[1:rows + 1, cols:] == CANARY).all(), what
