"""Exact rational helpers for pinning the oracle (test code only).

They restate the IEEE rules from first principles with Python integers and
``fractions.Fraction``: correctly rounded binary32 (ties to even, subnormals
included) and round-half-even to an integer. Nothing here calls the oracle.
"""
from fractions import Fraction
import struct

F32_MIN_EXP_Q = -149          # spacing of binary32 subnormals: 2^-149
F32_SIG_BITS = 24


def f32_value(x) -> Fraction:
    """Exact value of a binary32 number given as a Python/numpy float."""
    b = struct.pack("<f", float(x))
    (u,) = struct.unpack("<I", b)
    sign = -1 if u >> 31 else 1
    e = (u >> 23) & 0xFF
    frac = u & 0x7FFFFF
    if e == 0:
        return sign * Fraction(frac, 1 << 149)
    val = Fraction((1 << 23) | frac) * Fraction(2) ** (e - 150)
    return sign * val


def _floor_log2(a: Fraction) -> int:
    """floor(log2(a)) for a > 0."""
    n, d = a.numerator, a.denominator
    e = n.bit_length() - d.bit_length()
    # adjust so that 2^e <= a < 2^(e+1)
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_half_even(a: Fraction) -> int:
    """Nearest integer to a, ties to even."""
    f = a.numerator // a.denominator
    r = a - f
    if r > Fraction(1, 2):
        return f + 1
    if r < Fraction(1, 2):
        return f
    return f if f % 2 == 0 else f + 1


def round_to_f32(a: Fraction) -> Fraction:
    """Correctly rounded binary32 value of a rational (finite range assumed)."""
    if a == 0:
        return Fraction(0)
    sign = -1 if a < 0 else 1
    a = abs(a)
    e = _floor_log2(a)                       # 2^e <= a < 2^(e+1)
    q = max(e - (F32_SIG_BITS - 1), F32_MIN_EXP_Q)
    m = round_half_even(a / Fraction(2) ** q)
    return sign * Fraction(m) * Fraction(2) ** q


def quantize_exact(x: Fraction, s: Fraction) -> int:
    """round(x/s): the binary32 quotient rounded half-even to an integer,
    clamped to [-127, 127]; 0 when s == 0."""
    if s == 0:
        return 0
    quot = round_to_f32(x / s)
    q = round_half_even(quot)
    return max(-127, min(127, q))
