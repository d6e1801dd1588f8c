"""Pins the oracle's half-precision storage (binary16 and bfloat16 <->
binary32) and the typed GEMM / mean + SGD built on it, and its rolling hash.

Sources: "Verde与RepOps" §3.3 (IEEE-754 hardware needed; FP16 support limited)
and §5.3 (lower-precision training as future work); the ZKDV page's
proof.start (rolling_window hashes within each committed uint32 batch row).
The pages fix no format rules or hash; the library's definitions (exact
widening, one round-to-nearest-even narrowing; Rabin-Karp modulo 2^61 - 1 with
base 4294967311) are checked here against NumPy's float16 (an independent
implementation), exact rational rounding and Python integers.
"""
from fractions import Fraction

import numpy as np
import pytest

F32, F16, BF16 = 0, 1, 2
P = (1 << 61) - 1
BASE = 4294967311


def f32_of_bits(u):
    return np.array(u, dtype=np.uint32).view(np.float32)


def test_binary16_widening_all_patterns(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = orc.convert(h, F16, F32)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _narrow_cases():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = h[np.isfinite(h)].astype(np.float64)
    fin = np.unique(fin)
    mids = (fin[:-1] + fin[1:]) / 2                         # exact ties (representable in f32)
    mids32 = mids.astype(np.float32)
    up = np.nextafter(mids32, np.float32(np.inf))
    dn = np.nextafter(mids32, np.float32(-np.inf))
    rng = np.random.default_rng(0)
    rnd = (rng.standard_normal(200000) * np.exp2(rng.integers(-30, 20, 200000))).astype(np.float32)
    edge = np.array([65504, 65519.996, 65520, 65536, 1e30, -65520, 2.0 ** -24, 2.0 ** -25,
                     np.nextafter(np.float32(2.0 ** -25), np.float32(1)), 2.0 ** -26, 1e-40, -0.0, 0.0,
                     np.inf, -np.inf], dtype=np.float32)
    return np.concatenate([fin.astype(np.float32), mids32, up, dn, rnd, edge])


def test_binary16_narrowing_against_numpy(orc):
    x = _narrow_cases()
    got = orc.convert(x, F32, F16)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    n = orc.convert(np.array([np.nan], np.float32), F32, F16)
    assert np.isnan(n.view(np.float16)[0])


def bf16_value(b):
    """Exact value of a bfloat16 bit pattern, decoded by hand."""
    s = -1 if b >> 15 else 1
    e = (b >> 7) & 0xff
    m = b & 0x7f
    if e == 0:
        return s * Fraction(m, 1 << 7) * Fraction(1, 1 << 126)
    return s * (1 + Fraction(m, 1 << 7)) * Fraction(2) ** (e - 127)


def test_bfloat16_widening_exact(orc):
    b = np.array([0x0000, 0x8000, 0x3f80, 0xbf80, 0x0001, 0x007f, 0x0080, 0x7f7f, 0x4049, 0x1234],
                 dtype=np.uint16)
    got = orc.convert(b, BF16, F32)
    for v, bits in zip(got, b):
        assert Fraction(float(v)) == bf16_value(int(bits))
    assert np.isinf(orc.convert(np.array([0x7f80], np.uint16), BF16, F32)[0])
    assert np.isnan(orc.convert(np.array([0x7fc1], np.uint16), BF16, F32)[0])


def bf16_round(x):
    """Round-to-nearest-even of a finite float32 to bfloat16, in exact arithmetic."""
    v = Fraction(float(x))
    if v == 0:
        return 0x8000 if np.signbit(x) else 0
    best = None
    u = int(np.array(x, np.float32).view(np.uint32)) >> 16
    for c in (u - 1, u, u + 1, u + 2):           # the neighbours of the truncation
        c &= 0xffff
        if ((c >> 7) & 0xff) == 0xff:
            continue
        d = abs(bf16_value(c) - v)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0 and (best[1] & 1)):
            best = (d, c)
    return best[1]


def test_bfloat16_narrowing_exact_rational(orc):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(3000) * np.exp2(rng.integers(-140, 120, 3000))).astype(np.float32)
    ties = f32_of_bits((rng.integers(0, 1 << 15, 1000, dtype=np.uint32) << 16) | 0x8000)   # exact halfway
    x = np.concatenate([x, ties[np.isfinite(ties)], np.array([1e-45, -1e-45, 3.3895e38], np.float32)])
    got = orc.convert(x, F32, BF16)
    for xi, g in zip(x, got):
        if abs(float(xi)) >= 3.3895313892515355e38:    # rounds past the largest finite value
            assert (int(g) & 0x7fff) == 0x7f80
        else:
            assert int(g) == bf16_round(xi), (float(xi), hex(int(g)))
    assert (int(orc.convert(np.array([np.inf], np.float32), F32, BF16)[0])) == 0x7f80


@pytest.mark.parametrize("ta,tb,tc", [(F16, F16, F32), (BF16, BF16, F32), (BF16, F32, BF16), (F16, BF16, F16)])
def test_typed_gemm_is_the_widened_gemm_narrowed(orc, ta, tb, tc):
    rng = np.random.default_rng(10 * ta + tb)
    A32 = rng.standard_normal((13, 21)).astype(np.float32)
    B32 = rng.standard_normal((21, 9)).astype(np.float32)
    A = A32 if ta == F32 else orc.convert(A32, F32, ta)
    B = B32 if tb == F32 else orc.convert(B32, F32, tb)
    C = orc.gemm_typed(A, ta, B, tb, tc)
    Aw = A if ta == F32 else orc.convert(A, ta, F32)
    Bw = B if tb == F32 else orc.convert(B, tb, F32)
    C32 = orc.gemm(Aw, Bw)
    want = C32 if tc == F32 else orc.convert(C32, F32, tc)
    assert np.array_equal(C.view(np.uint16 if tc != F32 else np.uint32), want.view(C.dtype if tc != F32 else np.uint32))
    if ta == F16 and tb == F16:       # binary16 widening agrees with NumPy's
        C2 = orc.gemm(A.view(np.float16).astype(np.float32), B.view(np.float16).astype(np.float32))
        assert np.array_equal(C.view(np.uint32), C2.view(np.uint32))


def test_typed_mean_is_the_widened_mean(orc):
    rng = np.random.default_rng(3)
    g32 = [rng.standard_normal(1000).astype(np.float32) * 0.01 for _ in range(5)]
    order = [3, 1, 4, 0, 2]
    for t in (F16, BF16):
        gs = [orc.convert(g, F32, t) for g in g32]
        th = rng.standard_normal(1000).astype(np.float32)
        want = orc.mean_sgd([orc.convert(g, t, F32) for g in gs], order, 1e-3, th)
        got = orc.mean_sgd_typed(gs, t, order, 1e-3, th)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def ref_window(words, W):
    return [sum(int(w) * pow(BASE, W - 1 - t, P) for t, w in enumerate(words[i:i + W])) % P
            for i in range(len(words) - W + 1)]


@pytest.mark.parametrize("W", [1, 2, 7, 32])
def test_rolling_hash_brute_force(orc, W):
    rng = np.random.default_rng(W)
    x = rng.integers(0, 1 << 32, (3, 50), dtype=np.uint64).astype(np.uint32)
    x[0, :5] = 0xffffffff
    h = orc.rolling_hash(x, W)
    for r in range(3):
        assert [int(v) for v in h[r]] == ref_window(list(x[r]), W)


def test_rolling_hash_closed_forms(orc):
    z = np.zeros((2, 40), np.uint32)
    assert not orc.rolling_hash(z, 8).any()                        # all-zero windows
    x = np.arange(1, 41, dtype=np.uint32).reshape(1, 40)
    assert np.array_equal(orc.rolling_hash(x, 1)[0], x[0].astype(np.uint64))   # W = 1: the word
    one = np.zeros((1, 10), np.uint32)
    one[0, 4] = 1
    h = orc.rolling_hash(one, 3)[0]                                 # a single 1 at offset t of a window
    assert [int(v) for v in h] == [0, 0, 1, BASE, BASE * BASE % P, 0, 0, 0]
    two = np.array([[5, 7]], np.uint32)
    assert int(orc.rolling_hash(two, 2)[0, 0]) == 5 * BASE + 7       # two words: injective, below P
    assert orc.rolling_hash(np.zeros((1, 4), np.uint32), 5).shape == (1, 0)
