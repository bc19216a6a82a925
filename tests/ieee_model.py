"""Exact rational model of IEEE-754 binary32 addition and multiplication.

Used only to pin the oracle: values are decoded from their bit patterns into
exact fractions, added or multiplied exactly, and rounded to binary32 with
round-to-nearest, ties-to-even, with gradual underflow (subnormals kept) and
overflow to infinity. No hardware floating-point operation decides a result
here, so agreement with the oracle is evidence about the oracle, not about a
shared rounding unit.

Sign of an exact zero result (IEEE 754-2019, 6.3): a sum of operands of
opposite sign (or of +0 and -0) that is exactly zero is +0 under
round-to-nearest; x + x keeps the sign of x when x is zero; a product's zero
has the XOR of the operands' signs.
"""
from __future__ import annotations

import struct
from fractions import Fraction

_MIN_EXP = -126          # exponent of the smallest normal
_MANT = 23               # fraction bits
_QMIN = _MIN_EXP - _MANT  # -149: the subnormal quantum exponent
_MAX_FINITE = Fraction((1 << 24) - 1, 1) * Fraction(2) ** (127 - 23)

POS_INF = 0x7F800000
NEG_INF = 0xFF800000


def bits_of(x: float) -> int:
    """binary32 bits of a Python float that already holds a binary32 value."""
    return struct.unpack("<I", struct.pack("<f", x))[0]


def float_of(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def is_nan(b: int) -> bool:
    return (b & 0x7F800000) == 0x7F800000 and (b & 0x007FFFFF) != 0


def is_inf(b: int) -> bool:
    return (b & 0x7FFFFFFF) == 0x7F800000


def sign_of(b: int) -> int:
    return (b >> 31) & 1


def decode(b: int) -> Fraction:
    """Exact value of a finite binary32 bit pattern (zeros decode to 0)."""
    e = (b >> 23) & 0xFF
    m = b & 0x7FFFFF
    if e == 0xFF:
        raise ValueError("not finite")
    if e == 0:
        v = Fraction(m) * Fraction(2) ** _QMIN
    else:
        v = Fraction(m | (1 << 23)) * Fraction(2) ** (e - 127 - _MANT)
    return -v if sign_of(b) else v


def _pow2(k: int) -> Fraction:
    return Fraction(2) ** k


def round_to_bits(q: Fraction, zero_negative: bool = False) -> int:
    """Round an exact rational to binary32 (RN-even, subnormals, overflow to inf)."""
    if q == 0:
        return 0x80000000 if zero_negative else 0
    neg = q < 0
    a = -q if neg else q
    # e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if a < _pow2(e):
        e -= 1
    elif a >= _pow2(e + 1):
        e += 1
    qexp = max(e, _MIN_EXP) - _MANT          # exponent of one unit in the last place
    scaled = a / _pow2(qexp)
    whole = scaled.numerator // scaled.denominator
    frac = scaled - whole
    if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and (whole & 1)):
        whole += 1
    value = Fraction(whole) * _pow2(qexp)
    sign = 0x80000000 if neg else 0
    if value > _MAX_FINITE:
        return sign | 0x7F800000
    if whole == 0:
        return sign  # underflow to a signed zero
    # encode exactly
    if value < _pow2(_MIN_EXP):
        return sign | int(value / _pow2(_QMIN))           # subnormal
    e2 = value.numerator.bit_length() - value.denominator.bit_length()
    if value < _pow2(e2):
        e2 -= 1
    mant = int(value / _pow2(e2 - _MANT)) - (1 << _MANT)
    return sign | ((e2 + 127) << 23) | mant


def add(x: int, y: int) -> int:
    """binary32 x + y, round-to-nearest-even, as bit patterns (no NaN inputs)."""
    if is_nan(x) or is_nan(y):
        return 0x7FC00000
    if is_inf(x) or is_inf(y):
        if is_inf(x) and is_inf(y) and sign_of(x) != sign_of(y):
            return 0x7FC00000
        return x if is_inf(x) else y
    q = decode(x) + decode(y)
    if q == 0:
        both_neg_zero = (x == 0x80000000 and y == 0x80000000)
        return round_to_bits(q, zero_negative=both_neg_zero)
    return round_to_bits(q)


def mul(x: int, y: int) -> int:
    """binary32 x * y, round-to-nearest-even, as bit patterns (finite inputs)."""
    q = decode(x) * decode(y)
    neg = sign_of(x) ^ sign_of(y)
    if q == 0:
        return 0x80000000 if neg else 0
    r = round_to_bits(q)
    return r


def recip(w: int) -> int:
    """fl(1 / w) for a positive integer w."""
    return round_to_bits(Fraction(1, w))


def chain(column_bits: list[int]) -> int:
    """Ascending serial chain over one column: acc = c[0]; acc = acc + c[r]."""
    acc = column_bits[0]
    for b in column_bits[1:]:
        acc = add(acc, b)
    return acc
