"""Exact-rational IEEE-754 binary32 arithmetic for brute-force pins.

Every operation is carried out exactly on Python `Fraction`s and then rounded
once to binary32, round-to-nearest, ties-to-even, with gradual underflow.  It
shares nothing with the C oracle or the CUDA library, so agreement with it on
tiny inputs pins both the oracle's rounding and its operation order.

Only finite inputs are supported (the tests feed finite values).
"""
import math
import struct
from fractions import Fraction

_EMIN = -126            # smallest normal exponent
_P = 24                 # significand bits
_SUB_Q = Fraction(1, 2 ** 149)   # quantum of the subnormal range
_OVER = Fraction(2 ** 128)


def bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def from_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def is_f32(x: float) -> bool:
    return math.isnan(x) or struct.unpack("<f", struct.pack("<f", x))[0] == x


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_f32(x: Fraction, zero_sign: int = 0) -> float:
    """Nearest binary32 to the exact rational x (ties to even).

    zero_sign is the sign to give a result that is exactly zero (1 = negative)."""
    if x == 0:
        return -0.0 if zero_sign else 0.0
    neg = x < 0
    a = -x if neg else x
    e = _floor_log2(a)
    q = _SUB_Q if e < _EMIN else Fraction(2) ** (e - (_P - 1))
    t = a / q
    n = t.numerator // t.denominator
    rem = t - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * q
    if v >= _OVER:
        return -math.inf if neg else math.inf
    if v == 0:                          # underflow to zero keeps the sign
        return -0.0 if neg else 0.0
    r = float(v)                        # exact: at most 24 significant bits
    return -r if neg else r


def _sign(x: float) -> int:
    return 1 if math.copysign(1.0, x) < 0 else 0


def mul(a: float, b: float) -> float:
    return round_f32(Fraction(a) * Fraction(b), _sign(a) ^ _sign(b))


def add(a: float, b: float) -> float:
    # exact zero sum: -0 only when both addends are -0 (round-to-nearest)
    zs = 1 if (_sign(a) and _sign(b)) else 0
    return round_f32(Fraction(a) + Fraction(b), zs)


def sub(a: float, b: float) -> float:
    return add(a, -b)


def div(a: float, b: float) -> float:
    return round_f32(Fraction(a) / Fraction(b), _sign(a) ^ _sign(b))


def gemm_entry(arow, bcol) -> float:
    """sum = +0; for k in order: sum = fl(sum + fl(a_k * b_k))."""
    s = 0.0
    for a, b in zip(arow, bcol):
        s = add(s, mul(float(a), float(b)))
    return s
