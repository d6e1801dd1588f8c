"""Pins the oracle's operators for a Llama-style decoder: the k-windowed
(banded) batched GEMM of causal attention, the causal softmax backward, SiLU
and the SiLU-gated MLP (SwiGLU) with its backward, and rotary position
embeddings (frequencies, the cos/sin table, the rotation and its inverse).

Sources: "Verde与RepOps" §3.2 (the k-chain from +0 with k increasing, every
product and sum rounded on its own), §4.3 (Llama-style training as the
workload).  The pages fix none of these operators; the library's definitions
are restated here in exact rational arithmetic (tests/fp32_exact.py) with
independent indexing, and held against the float64 values of the mathematical
functions, closed forms and invariants.
"""
import math

import numpy as np
import pytest

import fp32_exact as fx

F32 = np.float32


def u32(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


# ------------------------------------------------------------ k window ----

def window_ref(A, B, k_lo, k_hi):
    """Row i's chain over [max(0, i - k_lo), min(K - 1, i + k_hi)], k
    increasing from +0 (open sides for -1): exact rational restatement."""
    M, K = A.shape
    N = B.shape[1]
    C = np.zeros((M, N), np.float32)
    for i in range(M):
        lo = 0 if k_lo < 0 else max(0, i - k_lo)
        hi = K - 1 if k_hi < 0 else min(K - 1, i + k_hi)
        for j in range(N):
            s = 0.0
            for k in range(lo, hi + 1):
                s = fx.add(s, fx.mul(float(A[i, k]), float(B[k, j])))
            C[i, j] = s
    return C


def run_window(orc, A, B, k_lo, k_hi, transA=False, transB=False):
    M, K = A.shape
    N = B.shape[1]
    As = np.ascontiguousarray(A.T if transA else A).reshape(-1)
    Bs = np.ascontiguousarray(B.T if transB else B).reshape(-1)
    C = np.zeros(M * N, np.float32)
    orc.gemm_batched(transA, transB, 1, M, N, K, As, M if transA else K, 0, Bs, K if transB else N, 0,
                     C, N, 0, k_lo=k_lo, k_hi=k_hi)
    return C.reshape(M, N)


@pytest.mark.parametrize("k_lo,k_hi", [(-1, 0), (0, -1), (-1, 2), (3, -1), (1, 1), (0, 0), (-1, 20), (20, -1)])
@pytest.mark.parametrize("trans", [(False, False), (True, False), (False, True)])
def test_window_brute_force(orc, k_lo, k_hi, trans):
    rng = np.random.default_rng(100 + 7 * k_lo + k_hi)
    A = (rng.standard_normal((9, 11)) * np.exp2(rng.integers(-6, 6, (9, 11)))).astype(F32)
    B = rng.standard_normal((11, 5)).astype(F32)
    got = run_window(orc, A, B, k_lo, k_hi, *trans)
    assert np.array_equal(u32(got), u32(window_ref(A, B, k_lo, k_hi)))


def test_window_open_on_both_sides_is_the_gemm(orc):
    rng = np.random.default_rng(5)
    A = rng.standard_normal((7, 13)).astype(F32)
    B = rng.standard_normal((13, 6)).astype(F32)
    assert np.array_equal(u32(run_window(orc, A, B, -1, -1)), u32(orc.gemm(A, B)))


def test_empty_window_is_the_epilogue_of_zero(orc):
    # rows 0..3 with k_lo = 0 and K = 2: rows 2, 3 start past the end
    A = np.ones((4, 2), F32)
    B = np.ones((2, 3), F32)
    C = np.full(12, 7.0, F32)
    bias = np.array([1.5, -2.0, 0.25], F32)
    orc.gemm_batched(0, 0, 1, 4, 3, 2, A.reshape(-1), 2, 0, B.reshape(-1), 3, 0, C, 3, 0, 2.0, bias, k_lo=0)
    C = C.reshape(4, 3)
    assert np.array_equal(C[2], bias) and np.array_equal(C[3], bias)
    assert np.array_equal(C[0], (F32(2) * F32(2) + bias).astype(F32))   # k = 0, 1
    assert np.array_equal(C[1], (F32(2) * F32(1) + bias).astype(F32))   # k = 1 only


def causal_probs(orc, S, first=0, seed=0):
    rng = np.random.default_rng(seed)
    return orc.softmax_rows_causal((rng.standard_normal((S, S + first)) * 2).astype(F32), first)


@pytest.mark.parametrize("first", [0, 3])
def test_window_equals_full_chain_over_zeros(orc, first):
    # P (causal softmax output) is +0 past each row's prefix: the window
    # k <= i + first (P V) and k >= i - first (P^T dO) give the full chain's bits
    S = 37
    P = causal_probs(orc, S, first, seed=first)
    V = np.random.default_rng(9).standard_normal((S + first, 8)).astype(F32)
    assert np.array_equal(u32(run_window(orc, P, V, -1, first)), u32(orc.gemm(P, V)))
    Pt = np.ascontiguousarray(P.T)                       # (S + first) x S: row i nonzero for k >= i - first
    dO = np.random.default_rng(10).standard_normal((S, 8)).astype(F32)
    assert np.array_equal(u32(run_window(orc, Pt, dO, first, -1)), u32(orc.gemm(Pt, dO)))


def test_window_never_reads_past_its_band(orc):
    # non-finite B rows outside a row's band change nothing in that row
    S = 12
    P = causal_probs(orc, S, 0, seed=2)
    V = np.random.default_rng(3).standard_normal((S, 4)).astype(F32)
    Vbad = V.copy()
    Vbad[S - 1] = np.inf                                 # only the last row's band holds k = S - 1
    good = run_window(orc, P, V, -1, 0)
    bad = run_window(orc, P, Vbad, -1, 0)
    assert np.array_equal(u32(bad[:S - 1]), u32(good[:S - 1]))
    assert np.isnan(orc.gemm(P, Vbad)[0]).all()          # the full chain meets 0 * inf


# ------------------------------------------------ causal softmax backward ----

def tree(vals):
    v = [float(x) for x in vals]
    while len(v) > 1:
        out = []
        for s in range(0, len(v), 32):
            acc = v[s]
            for x in v[s + 1:s + 32]:
                acc = fx.add(acc, x)
            out.append(acc)
        v = out
    return v[0]


@pytest.mark.parametrize("first,period,cols", [(0, None, 40), (2, 5, 9), (0, 3, 70)])
def test_causal_softmax_backward_exact(orc, first, period, cols):
    rows = 10
    rng = np.random.default_rng(cols + first)
    p = orc.softmax_rows_causal((rng.standard_normal((rows, cols)) * 2).astype(F32), first, period)
    dp = rng.standard_normal((rows, cols)).astype(F32)
    dp_masked = dp.copy()
    per = period or rows
    for i in range(rows):
        dp_masked[i, min(cols, first + i % per + 1):] = np.nan    # never read
    ds = orc.softmax_backward_causal(p, dp_masked, first, period)
    for i in range(rows):
        L = min(cols, first + i % per + 1)
        s = tree([fx.mul(float(dp[i, j]), float(p[i, j])) for j in range(L)])
        want = [fx.mul(float(p[i, j]), fx.sub(float(dp[i, j]), s)) for j in range(L)] + [0.0] * (cols - L)
        assert [fx.bits(float(v)) for v in ds[i]] == [fx.bits(v) for v in want], i


def test_causal_softmax_backward_against_float64(orc):
    rows = cols = 50
    rng = np.random.default_rng(4)
    p = orc.softmax_rows_causal((rng.standard_normal((rows, cols)) * 2).astype(F32), 0)
    dp = rng.standard_normal((rows, cols)).astype(F32)
    ds = orc.softmax_backward_causal(p, dp, 0)
    mask = np.tril(np.ones((rows, cols), bool))
    p64, d64 = p.astype(np.float64), np.where(mask, dp, 0).astype(np.float64)
    want = p64 * (d64 - (d64 * p64).sum(1, keepdims=True))
    assert np.max(np.abs(np.where(mask, ds - want, 0))) < 1e-6
    assert np.all(u32(ds)[~mask] == 0)                    # +0 past the prefix


# ------------------------------------------------------------- SwiGLU ----

def ref_silu(orc, x):
    e = orc.exp(-x)
    den = fx.add(1.0, e)
    return fx.mul(x, fx.div(1.0, den))


def test_silu_exact_composition(orc):
    xs = np.concatenate([np.linspace(-30, 30, 2001), [0.0, -0.0, 1e-30, -1e-30, 80, -80, 100, -88]]).astype(F32)
    for x in xs:
        assert fx.bits(orc.silu(float(x))) == fx.bits(ref_silu(orc, float(x))), float(x)


def test_silu_against_float64_and_limits(orc):
    for x in np.linspace(-20, 20, 4001).astype(F32):
        x64 = float(x)
        want = x64 / (1.0 + math.exp(-x64))
        assert abs(orc.silu(float(x)) - want) <= 1e-6 * abs(want) + 1e-30, x64
    assert fx.bits(orc.silu(0.0)) == 0
    assert orc.silu(100.0) == 100.0                       # sigma rounds to 1
    assert fx.bits(orc.silu(-200.0)) == 0x80000000        # exp overflows: sigma = +0, -200 * +0 = -0
    assert math.isnan(orc.silu(float("nan")))


def test_swiglu_exact_composition(orc):
    rng = np.random.default_rng(11)
    g = (rng.standard_normal(300) * 4).astype(F32)
    u = rng.standard_normal(300).astype(F32)
    h = orc.swiglu(g, u)
    want = np.array([fx.mul(ref_silu(orc, float(a)), float(b)) for a, b in zip(g, u)], F32)
    assert np.array_equal(u32(h), u32(want))


def ref_swiglu_bwd(orc, g, u, dh):
    sg = fx.div(1.0, fx.add(1.0, orc.exp(-g)))
    a = fx.mul(g, sg)
    du = fx.mul(dh, a)
    t = fx.mul(dh, u)
    d = fx.mul(sg, fx.add(1.0, fx.mul(g, fx.sub(1.0, sg))))
    return fx.mul(t, d), du


def test_swiglu_backward_exact_composition(orc):
    rng = np.random.default_rng(12)
    g = (rng.standard_normal(300) * 4).astype(F32)
    u = rng.standard_normal(300).astype(F32)
    dh = rng.standard_normal(300).astype(F32)
    dg, du = orc.swiglu_backward(g, u, dh)
    for i in range(300):
        wg, wu = ref_swiglu_bwd(orc, float(g[i]), float(u[i]), float(dh[i]))
        assert fx.bits(float(dg[i])) == fx.bits(wg) and fx.bits(float(du[i])) == fx.bits(wu), i


def test_swiglu_backward_against_float64(orc):
    rng = np.random.default_rng(13)
    g = (rng.standard_normal(2000) * 4).astype(F32)
    u = rng.standard_normal(2000).astype(F32)
    dh = rng.standard_normal(2000).astype(F32)
    dg, du = orc.swiglu_backward(g, u, dh)
    g64, u64, d64 = g.astype(np.float64), u.astype(np.float64), dh.astype(np.float64)
    sg = 1 / (1 + np.exp(-g64))
    assert np.max(np.abs(du - d64 * g64 * sg)) < 1e-5
    assert np.max(np.abs(dg - d64 * u64 * sg * (1 + g64 * (1 - sg)))) < 1e-5
    # the derivative against a central difference of the forward
    hstep = 1e-3
    fd = (g64 + hstep) / (1 + np.exp(-(g64 + hstep))) - (g64 - hstep) / (1 + np.exp(-(g64 - hstep)))
    assert np.max(np.abs(dg - d64 * u64 * fd / (2 * hstep))) < 1e-4


# -------------------------------------------------------------- rotary ----

LN_BASE = float(F32(math.log(500000.0)))


def test_rope_frequencies(orc):
    f = orc.rope_frequencies(32, LN_BASE)
    assert f[0] == 1.0
    for i in range(32):
        frac = fx.div(float(i), 32.0)
        x = fx.mul(frac, LN_BASE)
        want = orc.exp(-x)
        assert fx.bits(float(f[i])) == fx.bits(want), i
        assert abs(float(f[i]) - 500000.0 ** (-i / 32)) <= 2e-6 * 500000.0 ** (-i / 32), i
    f3 = orc.rope_frequencies(3, LN_BASE)                # pairs not a power of two: i/3 rounded
    assert fx.bits(float(f3[1])) == fx.bits(orc.exp(-fx.mul(fx.div(1.0, 3.0), LN_BASE)))


def half_ulp(v):
    return float(np.spacing(np.abs(F32(v)))) / 2


def check_table(c, s, pos, freq):
    a = pos[:, None].astype(np.float64) * freq[None, :].astype(np.float64)
    for got, want in ((c, np.cos(a)), (s, np.sin(a))):
        err = np.abs(got.astype(np.float64) - want)
        tol = np.spacing(np.abs(got)).astype(np.float64) / 2 * (1 + 1e-6) + 1e-300
        assert np.all(err <= tol), float(np.max(err / tol))
        # the rounded double result: equal to the float32 of the true value
        # except within ~1e-16 of a rounding boundary
        assert np.mean(got != want.astype(F32)) < 1e-4


def test_rope_table_against_float64(orc):
    freq = orc.rope_frequencies(32, LN_BASE)
    c, s = orc.rope_table(4096, freq)
    check_table(c, s, np.arange(4096), freq)
    assert np.all(u32(c[0]) == u32(np.ones(32, F32))) and np.all(u32(s[0]) == 0)


def test_rope_table_large_angles_and_quadrants(orc):
    # angle = p * 1 up to 2^20 rad: the reduction needs all three parts of pi/2
    freq = np.array([1.0, 0.5, F32(1 / 3), 2.0 ** -20], F32)
    c, s = orc.rope_table(1 << 14, freq)
    check_table(c, s, np.arange(1 << 14), freq)
    big = np.array([1.0], F32)
    ps = np.array([(1 << 20) - 1, 1 << 19, 123457, 710, 355, 11, 22, 33, 44], np.int64)
    for p in ps:
        cc, ss = orc.rope_table(int(p) + 1, big)
        check_table(cc[-1:], ss[-1:], np.array([p]), big)


def rot_ref(x0, x1, c, s, inverse):
    if not inverse:
        return fx.sub(fx.mul(x0, c), fx.mul(x1, s)), fx.add(fx.mul(x0, s), fx.mul(x1, c))
    return fx.add(fx.mul(x0, c), fx.mul(x1, s)), fx.sub(fx.mul(x1, c), fx.mul(x0, s))


@pytest.mark.parametrize("inverse", [False, True])
@pytest.mark.parametrize("first,period", [(0, None), (5, 3)])
def test_rope_exact_composition(orc, inverse, first, period):
    rows, heads, pairs = 7, 3, 4
    rng = np.random.default_rng(20 + first)
    freq = orc.rope_frequencies(pairs, LN_BASE)
    c, s = orc.rope_table(16, freq)
    x = rng.standard_normal((rows, heads * 2 * pairs + 3)).astype(F32)   # 3 columns past the heads
    y = orc.rope(x, heads, c, s, first, period, inverse)
    per = period or rows
    for r in range(rows):
        pos = first + r % per
        for h in range(heads):
            for i in range(pairs):
                col = h * 2 * pairs + 2 * i
                w0, w1 = rot_ref(float(x[r, col]), float(x[r, col + 1]), float(c[pos, i]), float(s[pos, i]),
                                 inverse)
                assert fx.bits(float(y[r, col])) == fx.bits(w0) and fx.bits(float(y[r, col + 1])) == fx.bits(w1)
        assert np.array_equal(u32(y[r, heads * 2 * pairs:]), u32(x[r, heads * 2 * pairs:]))


def test_rope_rotation_conventions(orc):
    # adjacent pairs rotate counter-clockwise by the angle: (1, 0) -> (c, s),
    # (0, 1) -> (-s, c); position 0 is the identity
    freq = orc.rope_frequencies(2, LN_BASE)
    c, s = orc.rope_table(9, freq)
    x = np.tile(np.array([[1.0, 0.0, 0.0, 1.0]], F32), (9, 1))
    y = orc.rope(x, 1, c, s)
    assert np.array_equal(u32(y[:, 0]), u32(c[:, 0])) and np.array_equal(u32(y[:, 1]), u32(s[:, 0]))
    # 0*c - 1*s: +0 - s, so -s except at position 0, where +0 - (+0) = +0
    assert np.array_equal(u32(y[1:, 2]), u32(-s[1:, 1])) and u32(y[:1, 2])[0] == 0
    assert np.array_equal(u32(y[:, 3]), u32(c[:, 1]))
    z = np.random.default_rng(1).standard_normal((1, 8)).astype(F32)
    assert np.array_equal(orc.rope(z, 2, c, s), z)


def test_rope_preserves_norms_and_inverts(orc):
    rng = np.random.default_rng(30)
    freq = orc.rope_frequencies(32, LN_BASE)
    c, s = orc.rope_table(2048, freq)
    x = rng.standard_normal((2048, 128)).astype(F32)
    y = orc.rope(x, 2, c, s)
    n0 = (x.astype(np.float64).reshape(2048, 64, 2) ** 2).sum(-1)
    n1 = (y.astype(np.float64).reshape(2048, 64, 2) ** 2).sum(-1)
    assert np.max(np.abs(n1 - n0) / (n0 + 1e-30)) < 1e-6
    back = orc.rope(y, 2, c, s, inverse=True)
    assert np.max(np.abs(back - x)) < 1e-5
    # the angle is applied at each row's position: rotation by p then by -q of
    # the same pair is a rotation by p - q (checked on the float64 values)
    a = np.arange(2048)[:, None] * freq[None, :].astype(np.float64)
    want0 = x[:, 0::2][:, :32] * np.cos(a) - x[:, 1::2][:, :32] * np.sin(a)
    assert np.max(np.abs(y[:, 0:64:2] - want0)) < 1e-5
