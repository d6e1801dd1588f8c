"""Pins the contributor-mean + SGD oracle and the contributor sort.

The method: "Zoo Per-LLM Chain Soundness" §2 Definition "Aggregation rule",
Lemma "Order independence within a batch"; §5 "Ordering subroutine" (sorted
DIDs, left fold), "Update step" (theta_t = theta_{t-1} - eta * gbar_t).
"""
import numpy as np
import pytest

import fp32_exact as fx


def _b(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def _hex(lst):
    return np.array([int(x, 16) for x in lst], dtype=np.uint32)


def test_one_contributor_is_plain_sgd(orc):
    rng = np.random.default_rng(1)
    g = rng.standard_normal(1000).astype(np.float32)
    th = rng.standard_normal(1000).astype(np.float32)
    eta = np.float32(1e-3)
    got = orc.mean_sgd([g], [0], float(eta), th)
    # |C| = 1: gbar = g / 1 = g; numpy float32 ops round once each
    want = th - eta * g
    assert np.array_equal(_b(got), _b(want))


def test_integer_gradients_exact_closed_form(orc):
    # small integers: the fold is exact, /16 is exact, eta = 2^-4 and integer
    # theta keep every step exact
    rng = np.random.default_rng(2)
    gs = [rng.integers(-1000, 1001, size=257).astype(np.float32) for _ in range(16)]
    th = rng.integers(-1000, 1001, size=257).astype(np.float32)
    got = orc.mean_sgd(gs, list(range(16)), 0.0625, th)
    tot = np.sum(np.stack(gs).astype(np.int64), axis=0)
    want = th.astype(np.float64) - 0.0625 * (tot / 16.0)
    assert np.array_equal(got.astype(np.float64), want)


def test_order_detector(orc, golden):
    case = golden["mean_order_detector"]
    gs = [np.array(g, np.float32) for g in case["grads"]]
    th = np.array(case["theta"], np.float32)
    outs = []
    for c in case["cases"]:
        got = orc.mean_sgd(gs, c["order"], case["eta"], th)
        assert np.array_equal(_b(got), _hex(c["expected_bits"]))
        outs.append(_b(got).tobytes())
    assert outs[0] != outs[1]


def test_fold_starts_at_first_gradient(orc, golden):
    case = golden["mean_fold_starts_at_first_gradient"]
    gs = [_hex(g).view(np.float32) for g in case["grads_bits"]]
    th = _hex(case["theta_bits"]).view(np.float32)
    eta = float(_hex([case["eta_bits"]]).view(np.float32)[0])
    got = orc.mean_sgd(gs, case["order"], eta, th)
    assert np.array_equal(_b(got), _hex(case["expected_bits"]))
    assert not np.array_equal(_b(got), _hex(case["zero_start_bits"]))


def test_divides_by_count(orc, golden):
    case = golden["mean_divides_by_count"]
    gs = [np.array(g, np.float32) for g in case["grads"]]
    got = orc.mean_sgd(gs, case["order"], case["eta"], np.array(case["theta"], np.float32))
    assert np.array_equal(_b(got), _hex(case["expected_bits"]))
    assert not np.array_equal(_b(got), _hex(case["reciprocal_reading_bits"]))


def test_sixteen_contributors_divide_equals_scale(orc):
    # 16 is a power of two: S/16 and S*0.0625 are the same real number, so the
    # page's (1/k)-scaling and the correctly rounded division agree bit for bit
    rng = np.random.default_rng(4)
    gs = [(rng.standard_normal(4096) * 1e-2).astype(np.float32) for _ in range(16)]
    th = (rng.standard_normal(4096) * 0.02).astype(np.float32)
    got = orc.mean_sgd(gs, list(range(16)), 1e-3, th)
    S = gs[0].copy()
    for g in gs[1:]:
        S = S + g
    want = th - np.float32(1e-3) * (S * np.float32(0.0625))
    assert np.array_equal(_b(got), _b(want))


@pytest.mark.parametrize("k,n", [(1, 5), (2, 9), (3, 17), (5, 11), (7, 30)])
def test_brute_force_exact_rational(orc, k, n):
    rng = np.random.default_rng(100 + k)
    gs = [(rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
          for _ in range(k)]
    th = rng.standard_normal(n).astype(np.float32)
    order = list(rng.permutation(k))
    eta = float(np.float32(1e-3))
    got = orc.mean_sgd(gs, order, eta, th)
    for e in range(n):
        S = float(gs[order[0]][e])
        for r in range(1, k):
            S = fx.add(S, float(gs[order[r]][e]))
        gbar = fx.div(S, float(k))
        want = fx.sub(float(th[e]), fx.mul(eta, gbar))
        assert fx.bits(float(got[e])) == fx.bits(want), e


def test_order_must_be_a_permutation(orc):
    g = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        orc.mean_sgd([g, g, g], [0, 1, 1], 1e-3, g)
    with pytest.raises(ValueError):
        orc.mean_sgd([g, g], [0, 2], 1e-3, g)


def test_sort_ids_is_unsigned_lexicographic(orc):
    rng = np.random.default_rng(7)
    ids = [rng.bytes(32) for _ in range(50)]
    ids += [b"did:key:z6Mk", b"did:key:z6MkA", b"did:key:", b"\xff", b"\x00\xff"]
    order = orc.sort_ids(ids)
    # Python orders bytes lexicographically by unsigned value, prefixes first
    want = sorted(range(len(ids)), key=lambda r: ids[r])
    assert order == want


def test_sort_ids_rejects_duplicates(orc):
    with pytest.raises(ValueError):
        orc.sort_ids([b"abc", b"abd", b"abc"])
