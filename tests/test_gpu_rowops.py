"""GPU parity of the order-fixed row operators (softmax, LayerNorm, RMSNorm,
GeLU) against the oracle, through the C ABI.

"Verde与RepOps" §3.2 (order-critical dimensions serial or with synchronised
threads), §4.3 (LayerNorm, GeLU, ERF).  Bar: bit-exact, for every kernel
variant (threads per row, runs per thread, the long-row kernel), aligned and
unaligned rows, and in place.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

# columns chosen to hit each kernel shape: 32, 64, 128, 256 threads x 1 run,
# 256 x 2, 256 x 4 runs per thread, and the long-row kernel
COLS = [1, 5, 32, 33, 1000, 2048, 4096, 8192, 8193, 16384, 16385, 32768, 40000]


def u32(a):
    return np.ascontiguousarray(a).view(np.uint32)


def rows_input(rows, cols, seed, scale=3.0, pad=0):
    x = inputs.normal((rows, cols + pad), scale, seed, DEV)
    return x[:, :cols] if pad else x


@pytest.mark.parametrize("cols", COLS)
def test_softmax_matches_oracle(rp, orc, cols):
    rows = 5 if cols <= 8192 else 3
    x = rows_input(rows, cols, 1000 + cols)
    y = rp.softmax_rows(x)
    assert np.array_equal(u32(y.cpu().numpy()), u32(orc.softmax_rows(x.cpu().numpy())))


@pytest.mark.parametrize("cols", COLS)
def test_layernorm_matches_oracle(rp, orc, cols):
    rows = 5 if cols <= 8192 else 3
    x = rows_input(rows, cols, 2000 + cols, 2.0)
    g = inputs.normal((cols,), 1.0, 3, DEV)
    b = inputs.normal((cols,), 1.0, 4, DEV)
    y = rp.layernorm_rows(x, g, b, 1e-5)
    want = orc.layernorm_rows(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy(), 1e-5)
    assert np.array_equal(u32(y.cpu().numpy()), u32(want))


@pytest.mark.parametrize("cols", COLS)
def test_rmsnorm_matches_oracle(rp, orc, cols):
    rows = 5 if cols <= 8192 else 3
    x = rows_input(rows, cols, 3000 + cols, 1.0)
    g = inputs.normal((cols,), 1.0, 5, DEV)
    y = rp.rmsnorm_rows(x, g, 1e-6)
    want = orc.rmsnorm_rows(x.cpu().numpy(), g.cpu().numpy(), 1e-6)
    assert np.array_equal(u32(y.cpu().numpy()), u32(want))


@pytest.mark.parametrize("cols", [7, 1000, 8195])
def test_unaligned_rows_and_in_place(rp, orc, cols):
    # ld = cols + 1: rows are not 16-byte aligned -> scalar loads, same bits
    x = rows_input(4, cols, 4000 + cols, 3.0, pad=1)
    want = orc.softmax_rows(x.cpu().numpy())
    assert np.array_equal(u32(rp.softmax_rows(x).cpu().numpy()), u32(want))
    g = inputs.normal((cols,), 1.0, 6, DEV)
    b = inputs.normal((cols,), 1.0, 7, DEV)
    want_ln = orc.layernorm_rows(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy(), 1e-5)
    z = x.clone()
    rp.layernorm_rows(z, g, b, 1e-5, out=z)            # in place
    assert np.array_equal(u32(z.cpu().numpy()), u32(want_ln))


@pytest.mark.parametrize("cols", [32769, 38437, 393216])
def test_unaligned_long_rows(rp, orc, cols):
    # rows past 32,768 values that are not 16-byte aligned: the long-row
    # kernel, whose shared buffer holds every run result of the row (it was
    # once sized for 1,025 runs whenever the rows were unaligned)
    x = rows_input(2, cols, 4500 + cols, 3.0, pad=1)
    xh = x.cpu().numpy()
    assert np.array_equal(u32(rp.softmax_rows(x).cpu().numpy()), u32(orc.softmax_rows(xh)))
    y = rp.softmax_rows(x, causal_first=cols - 2, causal_period=2)
    assert np.array_equal(u32(y.cpu().numpy()), u32(orc.softmax_rows_causal(xh, cols - 2, 2)))
    g = inputs.normal((cols,), 1.0, 8, DEV)
    b = inputs.normal((cols,), 1.0, 9, DEV)
    want = orc.layernorm_rows(xh, g.cpu().numpy(), b.cpu().numpy(), 1e-5)
    assert np.array_equal(u32(rp.layernorm_rows(x, g, b, 1e-5).cpu().numpy()), u32(want))
    want = orc.rmsnorm_rows(xh, g.cpu().numpy(), 1e-6)
    assert np.array_equal(u32(rp.rmsnorm_rows(x, g, 1e-6).cpu().numpy()), u32(want))


@pytest.mark.parametrize("n", [1, 7, 4096, (1 << 20) + 3])
def test_gelu_matches_oracle(rp, orc, n):
    x = inputs.normal((n,), 3.0, 5000 + n, DEV)
    y = rp.gelu(x)
    assert np.array_equal(u32(y.cpu().numpy()), u32(orc.gelu(x.cpu().numpy())))
    base = inputs.normal((n + 1,), 3.0, 6000 + n, DEV)
    xs = base[1:]                                        # 4-byte aligned only
    assert np.array_equal(u32(rp.gelu(xs).cpu().numpy()), u32(orc.gelu(xs.cpu().numpy())))
    xi = x.clone()
    rp.gelu(xi, out=xi)
    assert torch.equal(xi, y)


def test_closed_forms_on_gpu(rp):
    y = rp.softmax_rows(torch.full((3, 1000), 2.5, device=DEV))
    assert torch.all(y == torch.tensor(1.0, dtype=torch.float32) / 1000.0)
    b = torch.linspace(-1, 1, 300, device=DEV)
    g = torch.full((300,), 2.0, device=DEV)
    y = rp.layernorm_rows(torch.full((2, 300), 7.5, device=DEV), g, b, 1e-5)
    assert torch.equal(y, torch.stack([b, b]))


@pytest.mark.slow
def test_decoder_sized_workloads_sampled(rp, orc):
    T, D = inputs.DECODER_TOKENS, inputs.DECODER_DIM
    X = inputs.normal((T, D), 1.0, 100, DEV)
    g = inputs.normal((D,), 1.0, 101, DEV)
    b = inputs.normal((D,), 0.1, 102, DEV)
    Y = rp.layernorm_rows(X, g, b, 1e-5)
    R = rp.rmsnorm_rows(X, g, 1e-6)
    rows = [0, 1, 2047, T - 1]
    Xh = X[rows].cpu().numpy()
    assert np.array_equal(u32(Y[rows].cpu().numpy()),
                          u32(orc.layernorm_rows(Xh, g.cpu().numpy(), b.cpu().numpy(), 1e-5)))
    assert np.array_equal(u32(R[rows].cpu().numpy()), u32(orc.rmsnorm_rows(Xh, g.cpu().numpy(), 1e-6)))
    H = inputs.normal((T, 4 * D), 1.0, 103, DEV)          # MLP activations 4096 x 8192
    G = rp.gelu(H)
    assert np.array_equal(u32(G[rows].cpu().numpy()), u32(orc.gelu(H[rows].cpu().numpy())))
    S = inputs.normal((8 * T, T), 3.0, 104, DEV)          # 8 heads of 4096 x 4096 scores
    P = rp.softmax_rows(S)
    srows = [0, 4095, 4096, 8 * T - 1]
    assert np.array_equal(u32(P[srows].cpu().numpy()), u32(orc.softmax_rows(S[srows].cpu().numpy())))


# ragged column counts on 16-byte aligned rows (ld a multiple of 4): the staged
# kernels with a partial last chunk and a partial last run, at every shape
@pytest.mark.parametrize("cols,pad", [(33, 3), (1001, 3), (8193, 3), (16385, 3), (32767, 1)])
def test_staged_rows_with_ragged_columns(rp, orc, cols, pad):
    x = rows_input(3, cols, 7000 + cols, 2.0, pad=pad)
    xh = x.cpu().numpy()
    assert np.array_equal(u32(rp.softmax_rows(x).cpu().numpy()), u32(orc.softmax_rows(xh)))
    g = inputs.normal((cols,), 1.0, 8, DEV)
    b = inputs.normal((cols,), 1.0, 9, DEV)
    assert np.array_equal(u32(rp.layernorm_rows(x, g, b, 1e-5).cpu().numpy()),
                          u32(orc.layernorm_rows(xh, g.cpu().numpy(), b.cpu().numpy(), 1e-5)))
    assert np.array_equal(u32(rp.rmsnorm_rows(x, g, 1e-6).cpu().numpy()),
                          u32(orc.rmsnorm_rows(xh, g.cpu().numpy(), 1e-6)))


# gamma and beta that are not 16-byte aligned are read per element instead of
# being staged in shared memory: same bits
@pytest.mark.parametrize("cols", [64, 2048, 12000])
def test_norms_with_unaligned_parameters(rp, orc, cols):
    x = rows_input(4, cols, 8000 + cols, 2.0)
    gb = inputs.normal((2, cols + 1), 1.0, 10, DEV)
    g, b = gb[0, 1:], gb[1, 1:]
    xh, gh, bh = x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy()
    assert np.array_equal(u32(rp.layernorm_rows(x, g, b, 1e-5).cpu().numpy()),
                          u32(orc.layernorm_rows(xh, gh, bh, 1e-5)))
    assert np.array_equal(u32(rp.rmsnorm_rows(x, g, 1e-6).cpu().numpy()), u32(orc.rmsnorm_rows(xh, gh, 1e-6)))


# many more rows than resident CTAs: every CTA strides over rows with the
# next row's copy in flight
def test_persistent_row_loop(rp, orc):
    x = rows_input(5000, 256, 9000, 3.0)
    y = rp.softmax_rows(x)
    pick = [0, 1, 1215, 1216, 2431, 4999]
    assert np.array_equal(u32(y[pick].cpu().numpy()), u32(orc.softmax_rows(x[pick].cpu().numpy())))


# causal: every kernel shape, aligned and unaligned rows, in place, first = 0
# and first > 0 (a later query block), and first past the row (no mask)
@pytest.mark.parametrize("cols,pad", [(5, 0), (37, 3), (1000, 0), (2048, 0), (4095, 1), (4096, 0), (4096, 1),
                                      (4097, 3), (8193, 3), (16385, 3), (40000, 0)])
@pytest.mark.parametrize("first", [0, 700])
def test_causal_softmax_matches_oracle(rp, orc, cols, pad, first):
    rows = 6 if cols <= 8192 else 3
    x = rows_input(rows, cols, 11000 + cols + first, 3.0, pad=pad)
    want = orc.softmax_rows_causal(x.cpu().numpy(), first)
    assert np.array_equal(u32(rp.softmax_rows(x, causal_first=first).cpu().numpy()), u32(want))
    z = x.clone()
    rp.softmax_rows(z, out=z, causal_first=first)
    assert np.array_equal(u32(z.cpu().numpy()), u32(want))


@pytest.mark.parametrize("cols,first,period", [(300, 0, 300), (2048, 0, 2048), (130, 3, 50)])
def test_causal_softmax_many_rows(rp, orc, cols, first, period):
    # more rows than the persistent grid has warps: every warp runs several
    # rows of different prefix lengths
    rows = 7000
    x = rows_input(rows, cols, 14000 + cols, 3.0)
    got = rp.softmax_rows(x, causal_first=first, causal_period=period)
    pick = [0, 1, 2, 3, 607, 608, 2431, 4095, 6998, 6999]
    xp = x[pick].cpu().numpy()
    want = np.stack([orc.softmax_rows_causal(xp[k:k + 1], first + (r % period), 10 ** 9)[0]
                     for k, r in enumerate(pick)])
    assert np.array_equal(u32(got[pick].cpu().numpy()), u32(want))


def test_causal_softmax_ignores_masked_values(rp):
    x = rows_input(64, 64, 12000, 3.0)
    y = rp.softmax_rows(x, causal_first=0)
    x2 = x.clone()
    mask = torch.triu(torch.ones(64, 64, dtype=torch.bool, device=DEV), diagonal=1)
    x2[mask] = float("nan")
    assert torch.equal(rp.softmax_rows(x2, causal_first=0), y)
    assert torch.equal(rp.softmax_rows(x, causal_first=64), rp.softmax_rows(x))
    assert torch.equal(rp.softmax_rows(x, causal_first=1 << 62), rp.softmax_rows(x))


@pytest.mark.parametrize("cols,period", [(64, 16), (2048, 100), (40000, 3)])
def test_causal_softmax_with_period(rp, orc, cols, period):
    rows = 3 * period if cols <= 2048 else 6
    x = rows_input(rows, cols, 13000 + cols, 3.0)
    want = orc.softmax_rows_causal(x.cpu().numpy(), 5, period)
    got = rp.softmax_rows(x, causal_first=5, causal_period=period)
    assert np.array_equal(u32(got.cpu().numpy()), u32(want))


def same_bits_or_both_nan(got, want):
    """Equal bits wherever the oracle's value is not NaN; NaN where it is
    (NaN payloads are not pinned)."""
    got, want = np.asarray(got, dtype=np.float32), np.asarray(want, dtype=np.float32)
    nan = np.isnan(want)
    return bool(np.array_equal(np.isnan(got), nan) and np.array_equal(u32(got[~nan]), u32(want[~nan])))


def special_rows(cols, seed):
    """Rows of N(0, 3) values with infinities, huge values, NaNs at the start
    of a 32-value run (a NaN there hides the rest of that run from the max), an
    all -inf row and a row of one huge value among tiny ones."""
    g = np.random.default_rng(seed)
    x = (g.standard_normal((8, cols)) * 3.0).astype(np.float32)
    x[0, 5] = np.inf
    x[1, 7] = -np.inf
    x[2, 32] = np.nan
    x[2, 33] = 1000.0
    x[3, :] = -np.inf
    x[4, 64] = np.nan
    x[4, 65] = 200.0
    x[4, 3] = 150.0
    x[5, 10] = 3.0e38
    x[5, 11] = -3.0e38
    x[6, :] = 1e-30
    x[6, cols - 1] = 90.0
    x[7, 0] = np.nan
    return x


@pytest.mark.parametrize("cols", [96, 2048, 4096])
def test_softmax_special_values_match_oracle(rp, orc, cols):
    x = special_rows(cols, 15000 + cols)
    xd = torch.from_numpy(x).to(DEV)
    assert same_bits_or_both_nan(rp.softmax_rows(xd).cpu().numpy(), orc.softmax_rows(x))
    for first in (0, 40):
        want = orc.softmax_rows_causal(x, first)
        assert same_bits_or_both_nan(rp.softmax_rows(xd, causal_first=first).cpu().numpy(), want)


def test_gelu_special_values_match_oracle(rp, orc):
    v = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 3.0e38, -3.0e38, 1e-45, -1e-45, 10.0, -10.0,
                  5.9, -5.9, 100.0, -100.0, 1e-20], dtype=np.float32)
    x = np.concatenate([v, (np.random.default_rng(16000).standard_normal(4093) * 5).astype(np.float32)])
    got = rp.gelu(torch.from_numpy(x).to(DEV)).cpu().numpy()
    assert same_bits_or_both_nan(got, orc.gelu(x))


@pytest.mark.parametrize("cols", [96, 2048, 40000])
def test_norms_special_values_match_oracle(rp, orc, cols):
    # rows with infinities, NaN, overflowing squares, all-zero and constant rows,
    # on the staged kernels and (40000 columns) the long-row kernel
    x = special_rows(cols, 18000 + cols)
    x[3, :] = 0.0                         # variance 0: 1/sqrt(eps)
    x[6, :] = 7.0                         # constant row
    g = np.random.default_rng(18100 + cols).standard_normal(cols).astype(np.float32)
    b = np.random.default_rng(18200 + cols).standard_normal(cols).astype(np.float32)
    xd, gd, bd = (torch.from_numpy(a).to(DEV) for a in (x, g, b))
    assert same_bits_or_both_nan(rp.layernorm_rows(xd, gd, bd, 1e-5).cpu().numpy(),
                                 orc.layernorm_rows(x, g, b, 1e-5))
    assert same_bits_or_both_nan(rp.rmsnorm_rows(xd, gd, 1e-6).cpu().numpy(), orc.rmsnorm_rows(x, g, 1e-6))
