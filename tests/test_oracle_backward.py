"""Pins the oracle's backward operators: column sums, GeLU, RMSNorm and
softmax backward.

Sources: "Verde与RepOps" §3.2 (order-critical reductions in a fixed order),
§4.3 (training; LayerNorm, GeLU, ERF need reproducible forms).  The pages fix
none of these; the library's definitions are restated here step by step in
exact rational arithmetic (the 32-ary tree restated independently), and the
results are held against the float64 derivatives of the mathematical
functions.
"""
import math

import numpy as np
import pytest

import fp32_exact as fx

RUN = 32


def ref_tree(vals):
    v = [float(x) for x in vals]
    while len(v) > 1:
        v = [_fold(v[s:s + RUN]) for s in range(0, len(v), RUN)]
    return v[0]


def _fold(run):
    acc = run[0]
    for x in run[1:]:
        acc = fx.add(acc, x)
    return acc


def wide(rng, shape):
    v = (rng.uniform(-1, 1, shape) * np.exp2(rng.integers(-10, 10, shape))).astype(np.float32)
    v[rng.random(shape) < 0.05] = 0.0
    return v


@pytest.mark.parametrize("rows", [1, 2, 31, 33, 70, 1100])
def test_colsum_is_the_tree_over_rows(orc, rows):
    x = wide(np.random.default_rng(rows), (rows, 5))
    y = orc.colsum(x)
    for j in range(5):
        assert fx.bits(float(y[j])) == fx.bits(ref_tree(x[:, j]))


def test_colsum_integer_closed_form(orc):
    x = np.random.default_rng(1).integers(-1000, 1000, (3000, 7)).astype(np.float32)
    assert np.array_equal(orc.colsum(x).astype(np.int64), x.astype(np.int64).sum(0))


def ref_gelu_grad(x, orc):
    z = fx.mul(x, 0.707106769084930419921875)
    e = orc.erfc_pos(abs(z))
    phi2 = fx.sub(2.0, e) if z >= 0 else e
    cdf = fx.mul(0.5, phi2)
    a = -fx.mul(0.5, fx.mul(x, x))
    pdf = fx.mul(orc.exp(a), float(np.float32(0.3989422917366028)))
    return fx.add(cdf, fx.mul(x, pdf))


def test_gelu_grad_exact_composition(orc):
    xs = np.concatenate([np.linspace(-9, 9, 3001), [0.0, -0.0, 1e-30, -0.7517, 20, -20]]).astype(np.float32)
    for x in xs:
        assert fx.bits(orc.gelu_grad(float(x))) == fx.bits(ref_gelu_grad(float(x), orc)), float(x)


def test_gelu_grad_against_float64(orc):
    for x in np.linspace(-8, 8, 4001).astype(np.float32):
        x64 = float(x)
        want = 0.5 * math.erfc(-x64 / math.sqrt(2)) + x64 * math.exp(-0.5 * x64 * x64) / math.sqrt(2 * math.pi)
        assert abs(orc.gelu_grad(float(x)) - want) <= 2e-6 + 2e-6 * abs(want), x64
    assert abs(orc.gelu_grad(0.0) - 0.5) < 1e-6
    dy = np.random.default_rng(2).standard_normal(100).astype(np.float32)
    x = np.random.default_rng(3).standard_normal(100).astype(np.float32)
    got = orc.gelu_backward(x, dy)
    assert np.array_equal(got.view(np.uint32),
                          np.array([fx.mul(float(d), orc.gelu_grad(float(v))) for v, d in zip(x, dy)],
                                   np.float32).view(np.uint32))


def ref_rms_bwd_row(x, g, eps, dy):
    n = float(np.float32(len(x)))
    ms = fx.div(ref_tree([fx.mul(float(v), float(v)) for v in x]), n)
    inv = fx.div(1.0, float(np.float32(math.sqrt(fx.add(ms, eps)))))
    xh = [fx.mul(float(v), inv) for v in x]
    gy = [fx.mul(float(d), float(gg)) for d, gg in zip(dy, g)]
    c = fx.div(ref_tree([fx.mul(a, b) for a, b in zip(gy, xh)]), n)
    dx = [fx.mul(inv, fx.sub(a, fx.mul(b, c))) for a, b in zip(gy, xh)]
    p = [fx.mul(float(d), b) for d, b in zip(dy, xh)]
    return dx, p


@pytest.mark.parametrize("cols", [1, 3, 32, 45, 130])
def test_rmsnorm_backward_exact_composition(orc, cols):
    rng = np.random.default_rng(cols)
    x = rng.standard_normal((3, cols)).astype(np.float32)
    g = rng.standard_normal(cols).astype(np.float32)
    dy = rng.standard_normal((3, cols)).astype(np.float32)
    res = rng.standard_normal((3, cols)).astype(np.float32)
    eps = float(np.float32(1e-5))
    dx, p = orc.rmsnorm_backward(x, g, eps, dy)
    dxr, pr = orc.rmsnorm_backward(x, g, eps, dy, res)
    for i in range(3):
        wdx, wp = ref_rms_bwd_row(x[i], g, eps, dy[i])
        assert [fx.bits(float(v)) for v in dx[i]] == [fx.bits(v) for v in wdx]
        assert [fx.bits(float(v)) for v in p[i]] == [fx.bits(v) for v in wp]
        assert [fx.bits(float(v)) for v in dxr[i]] == [fx.bits(fx.add(a, float(b))) for a, b in zip(wdx, res[i])]
        assert np.array_equal(pr[i].view(np.uint32), p[i].view(np.uint32))


def test_rmsnorm_backward_against_float64(orc):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4, 300)).astype(np.float32)
    g = rng.standard_normal(300).astype(np.float32)
    dy = rng.standard_normal((4, 300)).astype(np.float32)
    dx, p = orc.rmsnorm_backward(x, g, 1e-5, dy)
    x64, g64, d64 = x.astype(np.float64), g.astype(np.float64), dy.astype(np.float64)
    inv = 1 / np.sqrt((x64 ** 2).mean(1, keepdims=True) + 1e-5)
    xh = x64 * inv
    gy = d64 * g64
    want = inv * (gy - xh * (gy * xh).mean(1, keepdims=True))
    assert np.max(np.abs(dx - want)) < 1e-5
    assert np.max(np.abs(p - d64 * xh)) < 1e-5
    # the gradient is orthogonal to x: sum_j dx_j x_j = 0 up to rounding
    assert np.max(np.abs((dx.astype(np.float64) * x64).sum(1))) < 1e-3


def ref_softmax_bwd_row(p, dp):
    s = ref_tree([fx.mul(float(a), float(b)) for a, b in zip(dp, p)])
    return [fx.mul(float(a), fx.sub(float(b), s)) for a, b in zip(p, dp)]


@pytest.mark.parametrize("cols", [1, 5, 32, 33, 100])
def test_softmax_backward_exact_composition(orc, cols):
    rng = np.random.default_rng(50 + cols)
    p = orc.softmax_rows((rng.standard_normal((3, cols)) * 2).astype(np.float32))
    dp = rng.standard_normal((3, cols)).astype(np.float32)
    ds = orc.softmax_backward(p, dp)
    for i in range(3):
        assert [fx.bits(float(v)) for v in ds[i]] == [fx.bits(v) for v in ref_softmax_bwd_row(p[i], dp[i])]


def test_softmax_backward_properties(orc):
    rng = np.random.default_rng(9)
    p = orc.softmax_rows((rng.standard_normal((5, 200)) * 2).astype(np.float32))
    dp = rng.standard_normal((5, 200)).astype(np.float32)
    ds = orc.softmax_backward(p, dp)
    p64, d64 = p.astype(np.float64), dp.astype(np.float64)
    want = p64 * (d64 - (d64 * p64).sum(1, keepdims=True))
    assert np.max(np.abs(ds - want)) < 1e-6
    assert np.max(np.abs(ds.astype(np.float64).sum(1))) < 1e-5       # sum_j p_j = 1
    pc = orc.softmax_rows_causal((rng.standard_normal((6, 6)) * 2).astype(np.float32), 0)
    dsc = orc.softmax_backward(pc, rng.standard_normal((6, 6)).astype(np.float32))
    assert np.all(dsc[np.triu_indices(6, 1)] == 0.0)                 # masked entries: signed zeros
