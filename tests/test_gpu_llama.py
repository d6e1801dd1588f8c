"""GPU parity of the Llama-style layer's operators against the oracle, through
the C ABI: the banded (k-windowed) attention GEMMs, the causal softmax
backward, SwiGLU and its backward, and the rotary embedding (frequencies,
table, rotation and inverse).

"Verde与RepOps" §3.2 (the k-chain), §4.3 (Llama-style training).  Bar:
bit-exact, for every tile configuration and loader, ragged sizes spanning
several tiles, in place and on column blocks of wider matrices.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
F32 = np.float32


def u32(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def bits(t):
    return u32(t.cpu().numpy())


def causal_probs(orc, S, cols, first, seed, period=None):
    x = inputs.normal((S, cols), 2.0, seed, "cpu").numpy()
    return orc.softmax_rows_causal(x, first, period)


# ------------------------------------------------------------ k window ----

@pytest.mark.parametrize("config,loader", list(itertools.product(range(5), (1, 2))))
def test_band_gemms_every_config(rp, orc, config, loader):
    # P V over k <= i + first (A = a causal softmax output), and P^T dO over
    # k >= i - first (A = its transpose, a strided view), 3 heads, ragged S
    S, first, d = 301, 2, 64
    P = np.stack([causal_probs(orc, S, S + first, first, 10 + h) for h in range(3)])
    V = inputs.normal((3, S + first, d), 1.0, 20, "cpu").numpy()
    want = np.stack([orc.gemm(P[h], V[h]) for h in range(3)])
    Pbuf = torch.zeros(3, S, 304, device=DEV)                   # a 16-byte row pitch: TMA can load P
    Pbuf[:, :, :S + first] = torch.from_numpy(P).to(DEV)
    Pd, Vd = Pbuf[:, :, :S + first], torch.from_numpy(V).to(DEV)
    got = rp.gemm_batched(Pd, Vd, k_hi=first, config=config, loader=loader)
    assert np.array_equal(bits(got), u32(want))
    dO = inputs.normal((3, S, d), 1.0, 21, "cpu").numpy()
    want_t = np.stack([orc.gemm(np.ascontiguousarray(P[h].T), dO[h]) for h in range(3)])
    got_t = rp.gemm_batched(Pd.transpose(1, 2), torch.from_numpy(dO).to(DEV), k_lo=first, config=config,
                            loader=loader)
    assert np.array_equal(bits(got_t), u32(want_t))


@pytest.mark.parametrize("config,loader", list(itertools.product(range(5), (1, 2))))
def test_grouped_b_every_config(rp, orc, config, loader):
    # 6 query heads over 2 key/value heads (groups of 3): Q K^T with K^T a
    # transposed view, then P V over the band k <= i
    H, G, S, d = 6, 3, 136, 64
    Q = inputs.normal((H, S, d), 1.0, 60, "cpu").numpy()
    K = inputs.normal((H // G, S, d), 1.0, 61, "cpu").numpy()
    Cs = np.zeros(H * S * S, F32)
    orc.gemm_batched(0, 1, H, S, S, d, Q.reshape(-1), d, S * d, K.reshape(-1), d, S * d, Cs, S, S * S, 0.125,
                     b_group=G)
    Kd = torch.from_numpy(K).to(DEV)
    got = rp.gemm_batched(torch.from_numpy(Q).to(DEV), Kd.transpose(1, 2), alpha=0.125, config=config,
                          loader=loader)
    assert np.array_equal(bits(got), u32(Cs.reshape(H, S, S)))
    P = np.stack([orc.softmax_rows_causal(Cs.reshape(H, S, S)[h], 0) for h in range(H)])
    V = inputs.normal((H // G, S, d), 1.0, 62, "cpu").numpy()
    Co = np.zeros(H * S * d, F32)
    orc.gemm_batched(0, 0, H, S, d, S, P.reshape(-1), S, S * S, V.reshape(-1), d, S * d, Co, d, S * d,
                     k_hi=0, b_group=G)
    got_o = rp.gemm_batched(torch.from_numpy(P).to(DEV), torch.from_numpy(V).to(DEV), k_hi=0, config=config,
                            loader=loader)
    assert np.array_equal(bits(got_o), u32(Co.reshape(H, S, d)))


def test_band_matches_the_oracle_window_with_epilogue(rp, orc):
    # the oracle's own window (chain over the band only) with alpha and an
    # in-place residual, and rows whose window is empty (k_lo with M > K)
    S = 200
    P = causal_probs(orc, S, S, 0, 30)
    V = inputs.normal((S, 48), 1.0, 31, "cpu").numpy()
    R = inputs.normal((S, 48), 1.0, 32, "cpu").numpy()
    C = R.reshape(-1).copy()
    orc.gemm_batched(0, 0, 1, S, 48, S, P.reshape(-1), S, 0, V.reshape(-1), 48, 0, C, 48, 0, 0.125, None, 0,
                     C, 48, 0, k_lo=-1, k_hi=0)
    Cd = torch.from_numpy(R).to(DEV)
    rp.gemm_batched(torch.from_numpy(P).to(DEV), torch.from_numpy(V).to(DEV), out=Cd, alpha=0.125, residual=Cd,
                    k_hi=0)
    assert np.array_equal(bits(Cd), u32(C.reshape(S, 48)))
    # 300 rows over K = 100 with k_lo = 0: rows >= 100 have no k left
    A = np.triu(inputs.normal((300, 100), 1.0, 33, "cpu").numpy())   # +0 below the diagonal
    B = inputs.normal((100, 40), 1.0, 34, "cpu").numpy()
    bias = inputs.normal((40,), 1.0, 35, "cpu").numpy()
    Cw = np.zeros(300 * 40, F32)
    orc.gemm_batched(0, 0, 1, 300, 40, 100, A.reshape(-1), 100, 0, B.reshape(-1), 40, 0, Cw, 40, 0, 1.0, bias,
                     k_lo=0)
    got = rp.gemm_batched(torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV),
                          bias=torch.from_numpy(bias).to(DEV), k_lo=0)
    assert np.array_equal(bits(got), u32(Cw.reshape(300, 40)))
    assert np.array_equal(bits(got)[100:], np.tile(u32(bias), (200, 1)))


def test_band_with_causal_output_skip(rp, orc):
    # dS K with dS from the causal backward (+0 past the diagonal) and scores
    # Q K^T with the output tile skip, together in one call each
    S, d = 260, 64
    P = causal_probs(orc, S, S, 0, 40)
    dP = inputs.normal((S, S), 1.0, 41, "cpu").numpy()
    dS = orc.softmax_backward_causal(P, dP, 0)
    K = inputs.normal((S, d), 1.0, 42, "cpu").numpy()
    want = (orc.gemm(dS, K) * F32(0.125)).astype(F32)
    got = rp.gemm_batched(torch.from_numpy(dS).to(DEV), torch.from_numpy(K).to(DEV), alpha=0.125, k_hi=0)
    assert np.array_equal(bits(got), u32(want))


# ------------------------------------------------ causal softmax backward ----

@pytest.mark.parametrize("rows,cols,first,period", [(96, 96, 0, None), (70, 333, 5, 35), (40, 9000, 0, 20),
                                                    (64, 64, 100, None)])
def test_causal_softmax_backward(rp, orc, rows, cols, first, period):
    x = inputs.normal((rows, cols), 2.0, rows + cols, "cpu").numpy()
    p = orc.softmax_rows_causal(x, first, period)
    dp = inputs.normal((rows, cols), 1.0, 7, "cpu").numpy()
    want = orc.softmax_backward_causal(p, dp, first, period)
    dp_dirty = dp.copy()
    per = period or rows
    for i in range(rows):
        dp_dirty[i, min(cols, first + i % per + 1):] = np.nan                      # never read
    pd, dd = torch.from_numpy(p).to(DEV), torch.from_numpy(dp_dirty).to(DEV)
    got = rp.softmax_backward(pd, dd, causal_first=first, causal_period=period)
    assert np.array_equal(bits(got), u32(want))
    rp.softmax_backward(pd, dd, out=dd, causal_first=first, causal_period=period)   # in place over dp
    assert np.array_equal(bits(dd), u32(want))


def test_causal_softmax_backward_unaligned_rows(rp, orc):
    # a pitch that is not a multiple of 4 takes the long-row kernel
    rows, cols = 50, 77
    p = orc.softmax_rows_causal(inputs.normal((rows, cols), 2.0, 3, "cpu").numpy(), 0)
    dp = inputs.normal((rows, cols), 1.0, 4, "cpu").numpy()
    want = orc.softmax_backward_causal(p, dp, 0)
    buf = torch.zeros(rows, 79, device=DEV)
    buf[:, :cols] = torch.from_numpy(dp).to(DEV)
    got = rp.softmax_backward(torch.from_numpy(p).to(DEV), buf[:, :cols], causal_first=0)
    assert np.array_equal(bits(got), u32(want))


# -------------------------------------------------------------- SwiGLU ----

def test_swiglu_matches_oracle(rp, orc):
    T, f = 130, 700
    gu = inputs.normal((T, 2 * f), 3.0, 50, "cpu").numpy()
    gu[0, :8] = [0.0, -0.0, 100.0, -100.0, -200.0, 90.0, -88.0, 1e-30]
    want = orc.swiglu(gu[:, :f], gu[:, f:])
    gd = torch.from_numpy(gu).to(DEV)
    got = rp.swiglu(gd[:, :f], gd[:, f:])                                    # column blocks, pitch 2f
    assert np.array_equal(bits(got), u32(want))
    out = gd[:, :f]
    rp.swiglu(gd[:, :f], gd[:, f:], out=out)                                 # in place over g
    assert np.array_equal(bits(gd[:, :f]), u32(want))


def test_swiglu_backward_matches_oracle(rp, orc):
    T, f = 97, 516
    gu = inputs.normal((T, 2 * f), 3.0, 60, "cpu").numpy()
    dh = inputs.normal((T, f), 1.0, 61, "cpu").numpy()
    wg, wu = orc.swiglu_backward(gu[:, :f], gu[:, f:], dh)
    gd, dd = torch.from_numpy(gu).to(DEV), torch.from_numpy(dh).to(DEV)
    dg, du = rp.swiglu_backward(gd[:, :f], gd[:, f:], dd)
    assert np.array_equal(bits(dg), u32(wg)) and np.array_equal(bits(du), u32(wu))
    # in place: dg over g and du over u, interleaved column blocks of one matrix
    rp.swiglu_backward(gd[:, :f], gd[:, f:], dd, dg=gd[:, :f], du=gd[:, f:])
    assert np.array_equal(bits(gd[:, :f]), u32(wg)) and np.array_equal(bits(gd[:, f:]), u32(wu))


def test_swiglu_scalar_path(rp, orc):
    # an odd width and pitch: no 16-byte accesses
    T, f = 33, 45
    g = inputs.normal((T, f), 3.0, 70, "cpu").numpy()
    u = inputs.normal((T, f), 1.0, 71, "cpu").numpy()
    buf = torch.zeros(T, f + 3, device=DEV)
    buf[:, :f] = torch.from_numpy(g).to(DEV)
    got = rp.swiglu(buf[:, :f], torch.from_numpy(u).to(DEV))
    assert np.array_equal(bits(got), u32(orc.swiglu(g, u)))


# -------------------------------------------------------------- rotary ----

LN_BASE = math.log(500000.0)


def test_rope_frequencies_and_table(rp, orc):
    for pairs in (32, 3, 64):
        f = rp.rope_frequencies(pairs, LN_BASE, DEV)
        want_f = orc.rope_frequencies(pairs, float(F32(LN_BASE)))
        assert np.array_equal(bits(f), u32(want_f))
        c, s = rp.rope_table(2048, f)
        wc, wsn = orc.rope_table(2048, want_f)
        assert np.array_equal(bits(c), u32(wc)) and np.array_equal(bits(s), u32(wsn))
    # large angles: frequency 1 out to position 2^20 - 1
    one = torch.tensor([1.0, 0.5, 2.0 ** -20], device=DEV)
    c, s = rp.rope_table(1 << 20, one)
    wc, wsn = orc.rope_table(1 << 20, one.cpu().numpy())
    assert np.array_equal(bits(c), u32(wc)) and np.array_equal(bits(s), u32(wsn))


@pytest.mark.parametrize("inverse", [False, True])
def test_rope_matches_oracle(rp, orc, inverse):
    # the query and key heads of a qkv matrix (40 of its 48 heads rotated),
    # positions repeating every 50 rows from 3 on
    rows, heads, pairs = 150, 40, 32
    freq = orc.rope_frequencies(pairs, float(F32(LN_BASE)))
    c, s = orc.rope_table(64, freq)
    x = inputs.normal((rows, 48 * 2 * pairs), 1.0, 80, "cpu").numpy()
    want = orc.rope(x, heads, c, s, 3, 50, inverse)
    xd = torch.from_numpy(x).to(DEV)
    rp.rope(xd, heads, torch.from_numpy(c).to(DEV), torch.from_numpy(s).to(DEV), first=3, period=50,
            inverse=inverse)
    assert np.array_equal(bits(xd), u32(want))


def test_rope_scalar_path_and_round_trip(rp, orc):
    # an odd pitch (no 8-byte accesses); forward then inverse is within
    # rounding of the identity
    rows, heads, pairs = 21, 3, 4
    freq = orc.rope_frequencies(pairs, float(F32(LN_BASE)))
    c, s = orc.rope_table(32, freq)
    x = inputs.normal((rows, heads * 2 * pairs + 1), 1.0, 90, "cpu").numpy()
    xd = torch.from_numpy(x).to(DEV)
    cd, sd = torch.from_numpy(c).to(DEV), torch.from_numpy(s).to(DEV)
    rp.rope(xd[:, 1:], heads, cd, sd)
    want_shift = orc.rope(x[:, 1:], heads, c, s)
    assert np.array_equal(bits(xd[:, 1:]), u32(want_shift)) and np.array_equal(bits(xd[:, 0]), u32(x[:, 0]))
    rp.rope(xd[:, 1:], heads, cd, sd, inverse=True)
    assert np.max(np.abs(xd.cpu().numpy() - x)) < 1e-5


def same_bits_or_both_nan(got, want):
    g, w = u32(got), u32(want)
    nan_g, nan_w = np.isnan(np.asarray(got, np.float32)), np.isnan(np.asarray(want, np.float32))
    return np.array_equal(nan_g, nan_w) and np.array_equal(g[~nan_g], w[~nan_w])


def test_special_values(rp, orc):
    # signed zeros, infinities, NaN, subnormals and overflow edges through
    # SwiGLU, its backward and the rotation (NaN payloads are not compared)
    sp = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 88.7, -88.7, 103.9, -103.9, 3e38, -3e38,
                   1.0, -1.0, 0.5], np.float32)
    g = np.tile(sp, (16, 1))
    u = np.tile(sp, (16, 1)).T.copy()
    gd, ud = torch.from_numpy(g).to(DEV), torch.from_numpy(u).to(DEV)
    assert same_bits_or_both_nan(rp.swiglu(gd, ud).cpu().numpy(), orc.swiglu(g, u))
    dh = np.roll(u, 3, axis=1)
    dg, du = rp.swiglu_backward(gd, ud, torch.from_numpy(dh).to(DEV))
    wg, wu = orc.swiglu_backward(g, u, dh)
    assert same_bits_or_both_nan(dg.cpu().numpy(), wg) and same_bits_or_both_nan(du.cpu().numpy(), wu)
    freq = orc.rope_frequencies(8, float(F32(LN_BASE)))
    c, s = orc.rope_table(16, freq)
    x = np.tile(sp, (16, 1))
    xd = torch.from_numpy(x).to(DEV)
    rp.rope(xd, 1, torch.from_numpy(c).to(DEV), torch.from_numpy(s).to(DEV))
    assert same_bits_or_both_nan(xd.cpu().numpy(), orc.rope(x, 1, c, s))
