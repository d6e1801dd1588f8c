"""Pins the order-fixed row operators of the oracle (softmax, LayerNorm,
RMSNorm, GeLU) and their building blocks (the 32-ary tree reduction, exp,
erfc).

Sources: "Verde与RepOps" §3.2 (order-critical dimensions run serially or with
synchronised threads), §3.3/§4.3 (LayerNorm, GeLU and ERF are the operators
behind DistilBERT's overhead).  The pages fix no algorithm; the library's
definitions (tree order, Cody-Waite exp, Numerical Recipes §6.2 erfc) are
restated here independently -- in exact rational arithmetic where the result is
a fixed sequence of roundings, against float64 libm where it approximates a
mathematical function.
"""
import math

import numpy as np
import pytest

import fp32_exact as fx

RUN = 32


def f32(x):
    return float(np.float32(x))


def ulp32(v: float) -> float:
    m, e = math.frexp(abs(v))
    return 2.0 ** max(e - 24, -149)


def ref_tree(vals, op):
    """The fixed 32-ary tree: fold runs of 32 left to right, level by level."""
    v = [float(x) for x in vals]
    while len(v) > 1:
        nxt = []
        for s in range(0, len(v), RUN):
            acc = v[s]
            for x in v[s + 1:s + RUN]:
                acc = fx.add(acc, x) if op == "sum" else (x if x > acc else acc)
            nxt.append(acc)
        v = nxt
    return v[0]


def _wide(rng, n):
    v = (rng.uniform(-1, 1, n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
    v[rng.random(n) < 0.05] = 0.0
    return v


@pytest.mark.parametrize("n", [1, 2, 5, 31, 32, 33, 64, 100, 1025, 1057])
def test_tree_sum_exact_rational(orc, n):
    v = _wide(np.random.default_rng(n), n)
    assert fx.bits(orc.row_sum(v)) == fx.bits(ref_tree(v, "sum"))


def test_tree_sum_order_detector(orc):
    # run 0 = [1e8, 1, -1e8, 1, 0 ...] folds to 1; a flat left fold over 64
    # values or a pairwise tree would give other values for the crafted row
    v = np.zeros(64, np.float32)
    v[:4] = [1e8, 1, -1e8, 1]
    v[32:36] = [1, 1e8, -1e8, 1]        # run 1: 1 + 1e8 -> 1e8, -1e8 -> 0, +1 -> 1
    assert orc.row_sum(v) == 2.0
    flat = np.float32(0)
    for x in v:
        flat = np.float32(flat + x)
    assert float(flat) == 1.0           # a flat left fold: 1 + 1e8 rounds away the 1
    w = np.ones(1000, np.float32)
    assert orc.row_sum(w) == 1000.0


def test_exp_accuracy_and_special_values(orc):
    xs = np.concatenate([np.linspace(-103.9, 88.72, 40001, dtype=np.float32),
                         np.random.default_rng(0).uniform(-30, 30, 20000).astype(np.float32)])
    worst = 0.0
    for x in xs:
        got, want = orc.exp(float(x)), math.exp(float(x))
        if want == 0.0 or math.isinf(want):
            continue
        worst = max(worst, abs(got - want) / ulp32(want))
    assert worst <= 1.5, worst
    assert orc.exp(0.0) == 1.0 and orc.exp(-0.0) == 1.0
    assert math.isnan(orc.exp(float("nan")))
    assert orc.exp(88.8) == math.inf and orc.exp(1000.0) == math.inf
    assert orc.exp(-104.0) == 0.0 and orc.exp(-1e30) == 0.0
    assert 0 < orc.exp(-100.0) < 2.0 ** -126          # a subnormal result
    assert abs(orc.exp(-100.0) - math.exp(-100.0)) <= 2.0 ** -149
    assert math.isfinite(orc.exp(88.72))


@pytest.mark.parametrize("lo,hi,bound", [(0, 1, 1e-6), (1, 2, 1.5e-6), (2, 4, 4e-6), (4, 6, 1e-5),
                                         (6, 10, 2e-5)])
def test_erfc_fit_accuracy(orc, lo, hi, bound):
    for z in np.linspace(lo, hi, 2001, dtype=np.float32):
        want = math.erfc(float(z))
        if want < 1e-37:
            continue
        assert abs(orc.erfc_pos(float(z)) - want) <= bound * want, z


@pytest.mark.parametrize("lo,hi,bound", [(-12, -6, 4e-5), (-6, -1, 8e-6), (-1, -0.01, 1e-6),
                                         (0.01, 1, 1e-6), (1, 12, 4e-7)])
def test_gelu_accuracy(orc, lo, hi, bound):
    x = np.linspace(lo, hi, 4001, dtype=np.float32)
    got = orc.gelu(x).astype(np.float64)
    x64 = x.astype(np.float64)
    ref = 0.5 * x64 * np.array([math.erfc(-t / math.sqrt(2)) for t in x64])
    m = ref != 0
    assert np.max(np.abs(got[m] - ref[m]) / np.abs(ref[m])) <= bound
    assert orc.gelu(np.zeros(1, np.float32))[0] == 0.0


def ref_softmax_row(row, orc):
    m = ref_tree(row, "max")
    e = [orc.exp(fx.sub(float(x), m)) for x in row]
    s = ref_tree(e, "sum")
    inv = fx.div(1.0, s)
    return [fx.mul(v, inv) for v in e]


@pytest.mark.parametrize("cols", [1, 7, 32, 33, 100, 257])
def test_softmax_exact_composition(orc, cols):
    rng = np.random.default_rng(cols)
    x = (rng.standard_normal((3, cols)) * 3).astype(np.float32)
    y = orc.softmax_rows(x)
    for i in range(3):
        want = ref_softmax_row(x[i], orc)
        assert [fx.bits(float(v)) for v in y[i]] == [fx.bits(v) for v in want]


def test_softmax_closed_forms(orc):
    for n in (1, 5, 32, 1000):
        y = orc.softmax_rows(np.full((2, n), 3.25, np.float32))
        assert np.all(y == np.float32(1) / np.float32(n))     # exp(0) = 1, sum = n, 1 * fl(1/n)
    # shifting an integer-valued row by an integer keeps x - max exact: same bits
    rng = np.random.default_rng(3)
    x = rng.integers(-20, 20, (4, 300)).astype(np.float32)
    assert np.array_equal(orc.softmax_rows(x).view(np.uint32), orc.softmax_rows(x + 1000).view(np.uint32))
    # close to the float64 softmax
    x = (rng.standard_normal((8, 500)) * 4).astype(np.float32)
    x64 = x.astype(np.float64)
    ref = np.exp(x64 - x64.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    assert np.max(np.abs(orc.softmax_rows(x) - ref) / ref) < 2e-6


def ref_layernorm_row(row, gamma, beta, eps):
    n = float(np.float32(len(row)))
    mean = fx.div(ref_tree(row, "sum"), n)
    d = [fx.sub(float(x), mean) for x in row]
    var = fx.div(ref_tree([fx.mul(v, v) for v in d], "sum"), n)
    denom = f32(math.sqrt(fx.add(var, eps)))   # double then float: innocuous double rounding
    inv = fx.div(1.0, denom)
    return [fx.add(fx.mul(fx.mul(v, inv), float(g)), float(b)) for v, g, b in zip(d, gamma, beta)]


@pytest.mark.parametrize("cols", [1, 2, 31, 64, 129])
def test_layernorm_exact_composition(orc, cols):
    rng = np.random.default_rng(40 + cols)
    x = (rng.standard_normal((2, cols)) * 2 + 1).astype(np.float32)
    g = rng.standard_normal(cols).astype(np.float32)
    b = rng.standard_normal(cols).astype(np.float32)
    eps = f32(1e-5)
    y = orc.layernorm_rows(x, g, b, eps)
    for i in range(2):
        want = ref_layernorm_row(x[i], g, b, eps)
        assert [fx.bits(float(v)) for v in y[i]] == [fx.bits(v) for v in want]


def test_layernorm_closed_forms_and_float64(orc):
    b = np.linspace(-1, 1, 300).astype(np.float32)
    g = np.full(300, 2.0, np.float32)
    y = orc.layernorm_rows(np.full((2, 300), 7.5, np.float32), g, b, 1e-5)
    assert np.array_equal(y, np.stack([b, b]))          # constant row: d = 0, y = beta
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((6, 2048)) * 3 + 2).astype(np.float32)
    g = rng.standard_normal(2048).astype(np.float32)
    b = rng.standard_normal(2048).astype(np.float32)
    x64 = x.astype(np.float64)
    mu = x64.mean(1, keepdims=True)
    ref = (x64 - mu) / np.sqrt(((x64 - mu) ** 2).mean(1, keepdims=True) + 1e-5) * g + b
    assert np.max(np.abs(orc.layernorm_rows(x, g, b, 1e-5) - ref)) < 2e-5


def ref_rmsnorm_row(row, gamma, eps):
    n = float(np.float32(len(row)))
    ms = fx.div(ref_tree([fx.mul(float(x), float(x)) for x in row], "sum"), n)
    denom = f32(math.sqrt(fx.add(ms, eps)))
    inv = fx.div(1.0, denom)
    return [fx.mul(fx.mul(float(x), inv), float(g)) for x, g in zip(row, gamma)]


@pytest.mark.parametrize("cols", [1, 3, 32, 65, 200])
def test_rmsnorm_exact_composition_and_float64(orc, cols):
    rng = np.random.default_rng(70 + cols)
    x = rng.standard_normal((2, cols)).astype(np.float32)
    g = rng.standard_normal(cols).astype(np.float32)
    eps = f32(1e-6)
    y = orc.rmsnorm_rows(x, g, eps)
    for i in range(2):
        assert [fx.bits(float(v)) for v in y[i]] == [fx.bits(v) for v in ref_rmsnorm_row(x[i], g, eps)]
    x64 = x.astype(np.float64)
    ref = x64 / np.sqrt((x64 ** 2).mean(1, keepdims=True) + 1e-6) * g
    assert np.max(np.abs(y - ref)) < 1e-5


def ref_exp(x: float) -> float:
    """The library's exp restated step by step (Cody-Waite reduction with a
    two-part ln 2, degree-7 Taylor polynomial by Horner's rule, scaling by
    2^k), every operation one binary32 rounding."""
    if x != x:
        return x
    if x > f32(88.72283935546875):
        return math.inf
    if x < f32(-103.972084045410156):
        return 0.0
    t = fx.mul(x, f32(1.44269502162933349609375))
    kf = float(round(t))                      # ties to even
    k = int(kf)
    r = fx.sub(x, fx.mul(kf, f32(0.693145751953125)))
    r = fx.sub(r, fx.mul(kf, f32(1.428606765330187045037746e-06)))
    p = f32(1.98412701e-04)
    for c in (1.38888892e-03, 8.33333377e-03, 4.16666679e-02, 1.66666672e-01, 0.5, 1.0, 1.0):
        p = fx.add(fx.mul(p, r), f32(c))
    if k > 127:
        return fx.mul(fx.mul(p, 2.0 ** 127), 2.0 ** (k - 127))
    if k < -126:
        return fx.mul(fx.mul(p, 2.0 ** (k + 64)), 2.0 ** -64)
    return fx.mul(p, 2.0 ** k)


def test_exp_steps_exact_rational(orc):
    rng = np.random.default_rng(12)
    xs = np.concatenate([rng.uniform(-104, 89, 3000), rng.uniform(-1, 1, 1000),
                         [0.0, -0.0, 88.72, -87.3, -100.0, -103.9, 0.34657359, -0.34657359]]).astype(np.float32)
    for x in xs:
        assert fx.bits(orc.exp(float(x))) == fx.bits(ref_exp(float(x))), float(x)


@pytest.mark.parametrize("first", [0, 3, 40])
def test_causal_softmax_is_the_prefix_softmax(orc, first):
    # row i sees keys 0 .. first + i: the softmax of that prefix, restated in
    # exact rational arithmetic, then +0
    rng = np.random.default_rng(100 + first)
    x = (rng.standard_normal((6, 37)) * 3).astype(np.float32)
    y = orc.softmax_rows_causal(x, first)
    for i in range(6):
        L = min(37, first + i + 1)
        want = ref_softmax_row(x[i, :L], orc) + [0.0] * (37 - L)
        assert [fx.bits(float(v)) for v in y[i]] == [fx.bits(v) for v in want]


def test_causal_softmax_closed_forms(orc):
    x = np.full((4, 9), 5.0, np.float32)
    y = orc.softmax_rows_causal(x, 0)
    for i in range(4):                      # a constant prefix of length i + 1: 1 * fl(1/(i+1))
        assert np.all(y[i, :i + 1] == np.float32(1) / np.float32(i + 1))
        assert np.all(y[i, i + 1:].view(np.uint32) == 0)
    x = np.random.default_rng(1).standard_normal((5, 33)).astype(np.float32)
    assert np.array_equal(orc.softmax_rows_causal(x, 1000).view(np.uint32), orc.softmax_rows(x).view(np.uint32))


def test_causal_softmax_period_repeats_the_block(orc):
    # period p: rows are blocks of p queries (one per head), each block masked
    # like the first
    x = (np.random.default_rng(2).standard_normal((12, 20)) * 2).astype(np.float32)
    y = orc.softmax_rows_causal(x, 2, period=4)
    for b in range(3):
        blk = slice(4 * b, 4 * b + 4)
        assert np.array_equal(y[blk].view(np.uint32), orc.softmax_rows_causal(x[blk], 2).view(np.uint32))
    assert np.array_equal(orc.softmax_rows_causal(x, 2, period=12).view(np.uint32),
                          orc.softmax_rows_causal(x, 2).view(np.uint32))
