"""Exact rational arithmetic for pinning the oracle.

`fl32` rounds an exact rational to the nearest binary32 (ties to even, with
the subnormal range), written from the IEEE-754 definition.  Tests use it to
evaluate the stated chain of single-rounded operations exactly and
independently of any floating-point unit, and compare with the exact real
result where the method's error bound applies."""
from fractions import Fraction

import numpy as np

EMIN = -126          # binary32 smallest normal exponent
MANT = 23            # binary32 fraction bits


def round_half_even(x: Fraction) -> int:
    """Nearest integer, ties to even."""
    f = x.numerator // x.denominator            # floor
    rem = x - f
    if rem > Fraction(1, 2):
        return f + 1
    if rem < Fraction(1, 2):
        return f
    return f if f % 2 == 0 else f + 1


def fl32(x: Fraction) -> Fraction:
    """Nearest binary32 to the rational x (no overflow handling needed here)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, EMIN)
    quantum = Fraction(2) ** (e - MANT)
    return sign * round_half_even(a / quantum) * quantum


def frac_of_f32(x) -> Fraction:
    return Fraction(float(np.float32(x)))


def frac_of_bf16_bits(h: int) -> Fraction:
    return Fraction(float(np.array([h << 16], dtype=np.uint32).view(np.float32)[0]))


def q_model(c: list[Fraction], qmax: int) -> tuple[list[int], Fraction]:
    """Codes and scale by the block rule evaluated exactly: scale = fl(m/qmax),
    inv = fl(qmax/m), q = clamp(rint(fl(c*inv)))."""
    m = max(abs(v) for v in c)
    if m < qmax * Fraction(2) ** EMIN:
        return [0] * len(c), Fraction(0)
    scale = fl32(m / qmax)
    inv = fl32(Fraction(qmax) / m)
    q = [max(-qmax, min(qmax, round_half_even(fl32(v * inv)))) for v in c]
    return q, scale


def unpack_int4(codes: np.ndarray) -> np.ndarray:
    """Signed int4 codes from packed bytes: element 2k is the low nibble of
    byte k, element 2k+1 the high nibble (two's complement)."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = (codes & 0x0F).astype(np.int8)
    hi = (codes >> 4).astype(np.int8)
    out = np.empty(codes.size * 2, dtype=np.int8)
    out[0::2] = lo
    out[1::2] = hi
    out[out >= 8] -= 16
    return out
