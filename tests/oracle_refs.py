"""Independent references used to pin the oracle (no import of oracle/ here).

* exact rational arithmetic (``fractions.Fraction``): the method's definition
  with exact sums, rounded exactly (round-to-nearest-even) at the rounding
  points the pages fix;
* integer matrix products (numpy int64) for the exact-integer special case.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

HALF = Fraction(1, 2)


def f32_to_frac(v) -> Fraction:
    return Fraction(float(np.float32(v)))


def bf16_bits_to_frac(h: int) -> Fraction:
    u = np.array([int(h) << 16], dtype=np.uint32).view(np.float32)[0]
    return Fraction(float(u))


def frac_to_bf16_bits(v: Fraction) -> int:
    """A Fraction exactly representable in BF16 -> its bit pattern."""
    f = np.array([float(v)], dtype=np.float32)
    assert Fraction(float(f[0])) == v, "not representable"
    u = int(f.view(np.uint32)[0])
    assert u & 0xFFFF == 0, "not a BF16 value"
    return u >> 16


def rne(v: Fraction, mant_bits: int, emin: int = -126) -> Fraction:
    """Round a rational to ``mant_bits`` significant bits, ties to even.

    ``emin`` is the smallest normal exponent; below it the spacing stays at
    2^(emin - mant_bits + 1) (gradual underflow). No overflow handling.
    """
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    q = Fraction(2) ** (e - (mant_bits - 1))
    t = a / q
    fl = t.numerator // t.denominator
    rem = t - fl
    if rem > HALF or (rem == HALF and fl % 2 == 1):
        fl += 1
    return sign * fl * q


def rne_bf16(v: Fraction) -> Fraction:
    return rne(v, 8)


def rne_f32(v: Fraction) -> Fraction:
    return rne(v, 24)


def exact_row(x_row, A, B, scale, base_row, max_rank, k_in, n_out, xa_given=None, d_given=None):
    """The fold of one routed row with exact sums and exact roundings.

    x_row, base_row: BF16 bits; A [max_rank, k_in], B [n_out, max_rank] BF16 bits;
    scale: f32. If ``xa_given`` / ``d_given`` (BF16 bits) are passed, the later
    stages start from them (stage-by-stage checking).
    Returns (xa_bits, xa_exact_sums, d_bits, d_exact_sums, out_bits).
    """
    xf = [bf16_bits_to_frac(v) for v in x_row]
    sums_xa, xa = [], []
    for c in range(max_rank):
        s = sum((xf[k] * bf16_bits_to_frac(A[c][k]) for k in range(k_in)), Fraction(0))
        sums_xa.append(s)
        xa.append(frac_to_bf16_bits(rne_bf16(s)))
    xa_use = list(xa_given) if xa_given is not None else xa
    xaf = [bf16_bits_to_frac(v) for v in xa_use]
    sums_d, d = [], []
    for j in range(n_out):
        s = sum((xaf[c] * bf16_bits_to_frac(B[j][c]) for c in range(max_rank)), Fraction(0))
        sums_d.append(s)
        d.append(frac_to_bf16_bits(rne_bf16(s)))
    d_use = list(d_given) if d_given is not None else d
    sc = f32_to_frac(scale)
    out = []
    for j in range(n_out):
        t = sc * bf16_bits_to_frac(d_use[j]) + bf16_bits_to_frac(base_row[j])
        out.append(frac_to_bf16_bits(rne_bf16(rne_f32(t))))   # fp32 fma, then BF16
    return xa, sums_xa, d, sums_d, out


def sum_is_unambiguous(exact: Fraction, abs_terms: Fraction, count: int, unit: Fraction) -> bool:
    """True if every value within the standard summation error bound of ``exact``
    rounds to the same BF16 value (so any summation order must agree)."""
    gamma = count * unit / (1 - count * unit)
    bound = gamma * abs_terms
    r = rne_bf16(exact)
    return rne_bf16(exact - bound) == r and rne_bf16(exact + bound) == r
