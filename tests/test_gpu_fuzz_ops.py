"""Seeded random parity cases for the decoder-step operators around the hot
path ("Verde与RepOps" §4.3, the Llama-style training step; §3.3 and §5.3,
half-precision storage; the ZKDV page's rolling windows): softmax backward
(plain and causal), RMSNorm backward with and without the residual path,
column sums, GeLU backward, SwiGLU and its backward on column blocks of one
matrix, the rotary rotation and its inverse, conversions between binary32,
binary16 and bfloat16, rolling hashes, and the batched GEMM with its
epilogue.

Shapes, leading-dimension padding, element offsets (misaligned rows), value
scales and in-place forms are drawn per case; every result must equal the
oracle's bit for bit (NaN where it is NaN), and outputs written into padded
buffers must leave the padding untouched.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CANARY = 9.75


def same(got, want, what):
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    if got.dtype.kind == "f":
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan), what
        got, want = got[~nan], want[~nan]
    assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), what


def padded(rng, rows, cols, seed, scale=1.0, fill=None):
    """(buffer, (rows, cols) view with padded pitch at a random element offset)."""
    pad, off = int(rng.integers(0, 6)), int(rng.integers(0, 4))
    ld = cols + pad
    if fill is None:
        buf = inputs.normal((off + rows * ld + 1,), scale, seed, DEV)
    else:
        buf = torch.full((off + rows * ld + 1,), fill, device=DEV)
    return buf, buf[off:off + rows * ld].view(rows, ld)[:, :cols]


def shape(rng, max_rows=400, max_cols=6000):
    rows = int(np.exp(rng.uniform(0.0, np.log(max_rows))))
    cols = int(np.exp(rng.uniform(0.0, np.log(max_cols))))
    return rows, cols


def host(t):
    return t.contiguous().cpu().numpy()


@pytest.mark.parametrize("case", range(60))
def test_random_softmax_backward(rp, orc, case):
    rng = np.random.default_rng(13_000 + case)
    rows, cols = shape(rng)
    _, x = padded(rng, rows, cols, 13_100 + case, 3.0)
    p = rp.softmax_rows(x)                               # a real probability matrix, contiguous
    _, dp = padded(rng, rows, cols, 13_200 + case)
    causal = bool(case % 2)
    first, period = int(rng.integers(0, cols)), int(rng.integers(1, rows + 1))
    if causal:
        p = rp.softmax_rows(x, causal_first=first, causal_period=period)
        want = orc.softmax_backward_causal(host(p), host(dp), first, period)
    else:
        want = orc.softmax_backward(host(p), host(dp))
    in_place = bool(rng.integers(2))
    if in_place:
        out = dp
    else:
        obuf, out = padded(rng, rows, cols, 0, fill=CANARY)
        before = obuf.clone()
    kw = dict(causal_first=first, causal_period=period) if causal else {}
    rp.softmax_backward(p, dp, out=out, **kw)
    torch.cuda.synchronize()
    what = dict(rows=rows, cols=cols, causal=causal, in_place=in_place)
    same(host(out), want, what)
    if not in_place:
        # only the view's elements may change: the padding and the slack stay canaries
        view_idx = torch.zeros_like(obuf, dtype=torch.bool)
        base = (out.data_ptr() - obuf.data_ptr()) // 4
        view_idx[base:base + rows * out.stride(0)].view(rows, out.stride(0))[:, :cols] = True
        assert ((obuf != before) & ~view_idx).sum().item() == 0, what
        assert (obuf[~view_idx] == CANARY).all(), what


@pytest.mark.parametrize("case", range(40))
def test_random_rmsnorm_backward_and_colsum(rp, orc, case):
    rng = np.random.default_rng(14_000 + case)
    rows, cols = shape(rng, 300, 12_000)
    _, x = padded(rng, rows, cols, 14_100 + case, 2.0)
    _, dy = padded(rng, rows, cols, 14_200 + case, 0.5)
    gamma = inputs.normal((cols,), 1.0, 14_300 + case, DEV)
    mode = case % 3                                      # 0: no residual, 1: a residual, 2: residual in dx
    res = None
    if mode:
        _, res = padded(rng, rows, cols, 14_400 + case)
    want_dx, want_p = orc.rmsnorm_backward(host(x), host(gamma), 1e-6, host(dy),
                                           host(res) if res is not None else None)
    if mode == 2:
        dx, dyxh = rp.rmsnorm_backward(x, gamma, 1e-6, dy, dx=res, res=res)
    else:
        dx, dyxh = rp.rmsnorm_backward(x, gamma, 1e-6, dy, res=res)
    torch.cuda.synchronize()
    what = dict(rows=rows, cols=cols, mode=mode)
    same(host(dx), want_dx, what)
    same(host(dyxh), want_p, what)
    # dgamma: column sums over the rows, from a padded view
    same(host(rp.colsum(dyxh)), orc.colsum(want_p), what)
    _, big = padded(rng, int(rng.integers(1, 3000)), int(rng.integers(1, 700)), 14_500 + case)
    same(host(rp.colsum(big)), orc.colsum(host(big)), what)


@pytest.mark.parametrize("case", range(40))
def test_random_elementwise_gelu_swiglu(rp, orc, case):
    rng = np.random.default_rng(15_000 + case)
    rows, cols = shape(rng, 300, 9000)
    scale = float(rng.choice([0.5, 3.0, 30.0]))
    # GeLU backward on a contiguous range at a random offset
    n = rows * cols
    off = int(rng.integers(0, 4))
    xb = inputs.normal((n + off,), scale, 15_100 + case, DEV)[off:]
    dyb = inputs.normal((n + off,), 1.0, 15_200 + case, DEV)[off:]
    same(host(rp.gelu_backward(xb, dyb)), orc.gelu_backward(host(xb), host(dyb)), ("gelu'", n))
    # SwiGLU on [g | u] column blocks of one padded matrix, then its backward
    _, gu = padded(rng, rows, 2 * cols, 15_300 + case, scale)
    g, u = gu[:, :cols], gu[:, cols:]
    want_h = orc.swiglu(host(g), host(u))
    h = rp.swiglu(g, u)
    _, dh = padded(rng, rows, cols, 15_400 + case)
    want_dg, want_du = orc.swiglu_backward(host(g), host(u), host(dh))
    dg, du = rp.swiglu_backward(g, u, dh)
    torch.cuda.synchronize()
    what = dict(rows=rows, cols=cols, scale=scale)
    same(host(h), want_h, what)
    same(host(dg), want_dg, what)
    same(host(du), want_du, what)
    # in place over g and u (the decoder's forms)
    rp.swiglu_backward(g, u, dh, dg=g, du=u)
    torch.cuda.synchronize()
    same(host(g), want_dg, what)
    same(host(u), want_du, what)


@pytest.mark.parametrize("case", range(40))
def test_random_rotary(rp, orc, case):
    rng = np.random.default_rng(16_000 + case)
    pairs = int(rng.integers(1, 65))
    heads = int(rng.integers(1, 9))
    rows = int(rng.integers(1, 600))
    period = int(rng.integers(1, rows + 1))
    first = int(rng.integers(0, 200))
    positions = first + period
    ln_base = float(np.log(rng.choice([10_000.0, 500_000.0])))
    freq = rp.rope_frequencies(pairs, ln_base)
    cos, sin = rp.rope_table(positions, freq)
    wf = orc.rope_frequencies(pairs, ln_base)
    wc, ws = orc.rope_table(positions, wf)
    same(host(freq), wf, "freq")
    same(host(cos), wc, "cos")
    same(host(sin), ws, "sin")
    extra = int(rng.integers(0, 5))
    _, x = padded(rng, rows, heads * 2 * pairs + extra, 16_100 + case)
    inverse = bool(case % 2)
    want = orc.rope(host(x), heads, wc, ws, first=first, period=period, inverse=inverse)
    rp.rope(x, heads, cos, sin, first=first, period=period, inverse=inverse)
    torch.cuda.synchronize()
    same(host(x), want, dict(pairs=pairs, heads=heads, rows=rows, period=period, first=first, inverse=inverse))


@pytest.mark.parametrize("case", range(40))
def test_random_conversions_and_rolling_hash(rp, orc, case):
    rng = np.random.default_rng(17_000 + case)
    n = int(np.exp(rng.uniform(0.0, np.log(3_000_000))))
    off = int(rng.integers(0, 4))
    scale = float(10.0 ** rng.uniform(-8, 6))
    x = inputs.normal((n + off,), scale, 17_100 + case, DEV)[off:]
    for dt, t in ((torch.float16, 1), (torch.bfloat16, 2)):
        h = rp.convert(x, dt)
        hb = h.view(torch.int16).cpu().numpy().view(np.uint16)
        same(hb, orc.convert(host(x), 0, t), ("narrow", dt, n))
        back = rp.convert(h, torch.float32)
        same(host(back), orc.convert(hb, t, 0), ("widen", dt, n))
    rows = int(rng.integers(1, 64))
    width = int(np.exp(rng.uniform(0.0, np.log(20_000))))
    window = int(rng.integers(1, width + 1)) if case % 2 else int(rng.integers(1, min(width, 40) + 1))
    rows = max(1, min(rows, int(3e7) // max(1, width * min(window, width - window + 1))))   # oracle time
    g = torch.Generator(device=DEV).manual_seed(17_200 + case)
    pad = int(rng.integers(0, 5))
    words = torch.randint(-2**31, 2**31 - 1, (rows, width + pad), generator=g, dtype=torch.int32,
                          device=DEV)[:, :width]
    got = rp.rolling_hash(words, window)
    want = orc.rolling_hash(words.contiguous().cpu().numpy().view(np.uint32), window)
    same(host(got).view(np.uint64), want, dict(rows=rows, width=width, window=window))


@pytest.mark.parametrize("case", range(60))
def test_random_batched_gemm_epilogue(rp, orc, case):
    rng = np.random.default_rng(18_000 + case)
    batch = int(rng.integers(1, 7))
    M, N, K = (int(np.exp(rng.uniform(0.0, np.log(300.0)))) for _ in range(3))
    alpha = float(np.float32(rng.choice([1.0, 0.125, -0.7])))
    use_bias, use_res, act = bool(rng.integers(2)), int(rng.integers(3)), int(rng.integers(2))
    ta, tb = bool(rng.integers(2)), bool(rng.integers(2))
    shared_b = bool(rng.integers(2))
    A = inputs.normal((batch, K, M) if ta else (batch, M, K), 1.0, 18_100 + case, DEV)
    A = A.transpose(1, 2) if ta else A
    nb = 1 if shared_b else batch
    B = inputs.normal((nb, N, K) if tb else (nb, K, N), 1.0, 18_200 + case, DEV)
    B = B.transpose(1, 2) if tb else B
    Bop = B[0] if shared_b else B
    bias = inputs.normal((N,), 1.0, 18_300 + case, DEV) if use_bias else None
    out = torch.full((batch, M, N), CANARY, device=DEV)
    R = None
    if use_res == 1:
        R = inputs.normal((batch, M, N), 1.0, 18_400 + case, DEV)
    elif use_res == 2:
        out = inputs.normal((batch, M, N), 1.0, 18_500 + case, DEV)
        R = out                                          # residual in place
    Rh = host(R) if R is not None else None
    rp.gemm_batched(A, Bop, out=out, alpha=alpha, bias=bias, act=act, residual=R)
    torch.cuda.synchronize()
    want = np.empty((batch, M, N), np.float32)
    for b in range(batch):
        Ab = np.ascontiguousarray(host(A[b]))
        Bb = np.ascontiguousarray(host(Bop if shared_b else B[b]))
        C = np.zeros(M * N, np.float32)
        orc.gemm_batched(0, 0, 1, M, N, K, Ab.reshape(-1), K, 0, Bb.reshape(-1), N, 0, C, N, 0, alpha=alpha,
                         bias=host(bias) if bias is not None else None, act=act,
                         R=Rh[b].reshape(-1) if Rh is not None else None, ldr=N)
        want[b] = C.reshape(M, N)
    same(host(out), want, dict(batch=batch, M=M, N=N, K=K, alpha=alpha, bias=use_bias, res=use_res, act=act,
                               ta=ta, tb=tb, shared_b=shared_b))


@pytest.mark.parametrize("case", range(60))
def test_random_batched_causal_and_banded(rp, orc, case):
    # interleaved heads (batch matrices as column blocks of one matrix),
    # B shared by groups of consecutive batches, then either a causal tile
    # skip (only elements on or below the boundary are defined) or a k band
    # per row with A +0 outside it (the attention products)
    rng = np.random.default_rng(23_000 + case)
    groups = int(rng.integers(1, 4))
    group = int(rng.integers(1, 4))
    batch = groups * group
    M = int(np.exp(rng.uniform(0.0, np.log(400.0))))
    N = int(np.exp(rng.uniform(0.0, np.log(200.0))))
    K = int(np.exp(rng.uniform(0.0, np.log(400.0))))
    X = inputs.normal((M, batch * K + 4), 1.0, 23_100 + case, DEV)
    A = X[:, :batch * K].view(M, batch, K).transpose(0, 1)          # (batch, M, K), stride K apart
    Bm = inputs.normal((groups, K, N), 1.0, 23_200 + case, DEV)
    banded = bool(case % 2)
    first, k_lo, k_hi = -1, -1, -1
    if banded:
        k_lo = int(rng.integers(0, K + 1)) if rng.integers(3) else -1
        k_hi = int(rng.integers(0, K + 1)) if (rng.integers(3) or k_lo < 0) else -1
        i = torch.arange(M, device=DEV)[:, None]
        k = torch.arange(K, device=DEV)[None, :]
        inside = torch.ones((M, K), dtype=torch.bool, device=DEV)
        if k_lo >= 0:
            inside &= k >= i - k_lo
        if k_hi >= 0:
            inside &= k <= i + k_hi
        A.mul_(inside.to(torch.float32))                                # +0 (or -0) outside each row's band
    else:
        first = int(rng.integers(0, max(1, N)))
    out = torch.full((batch, M, N), CANARY, device=DEV)
    rp.gemm_batched(A, Bm, out=out, causal_first=first, k_lo=k_lo, k_hi=k_hi)
    torch.cuda.synchronize()
    Ah = np.ascontiguousarray(host(X)[:, :batch * K])
    want = np.zeros(batch * M * N, np.float32)
    orc.gemm_batched(0, 0, batch, M, N, K, Ah.reshape(-1), batch * K, K, host(Bm).reshape(-1), N, K * N,
                     want, N, M * N, k_lo=k_lo, k_hi=k_hi, b_group=group)
    want = want.reshape(batch, M, N)
    got = host(out)
    what = dict(batch=batch, group=group, M=M, N=N, K=K, first=first, k_lo=k_lo, k_hi=k_hi)
    if first >= 0:
        defined = np.arange(N)[None, :] <= first + np.arange(M)[:, None]
        assert np.array_equal(got[:, defined].view(np.uint32), want[:, defined].view(np.uint32)), what
    else:
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), what
