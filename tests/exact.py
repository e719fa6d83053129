"""Exact-rational restatement of the codec's rounding steps, for brute-force pins.

Numbers are ``fractions.Fraction``; every rounding is written out from the definition
of round-to-nearest, ties-to-even onto a floating-point grid (the grid's spacing and
range are the only format parameters). Nothing here calls the oracle or the CUDA path,
and nothing here uses hardware floating-point arithmetic, so agreement with the oracle
pins the oracle's use of binary32 division, multiplication, addition and its BF16,
E4M3 and E8M0 encoders.
"""
from __future__ import annotations

from fractions import Fraction as F


def _round_half_even(r: F) -> int:
    return round(r)  # Fraction.__round__ rounds halves to the even integer


def round_to_grid(x: F, mant_bits: int, emin: int, emax: int, sat_max: F | None = None,
                  overflow_to_inf: bool = True):
    """Round x to the binary format with `mant_bits` fraction bits, normal exponents in
    [emin, emax] (subnormals below 2^emin with spacing 2^(emin - mant_bits)).

    Returns a Fraction, or the string 'inf'/'-inf' on overflow.
    """
    if x == 0:
        return F(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    elif F(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    quantum = F(2) ** (e - mant_bits)
    r = _round_half_even(a / quantum) * quantum
    largest = (2 - F(2) ** (-mant_bits)) * F(2) ** emax
    if sat_max is not None:
        if r > sat_max:
            r = sat_max
    elif r > largest:
        if overflow_to_inf:
            return "inf" if sign > 0 else "-inf"
    return sign * r


def f32(x: F) -> F:
    """Round to IEEE binary32 (24-bit significand, exponents -126..127)."""
    r = round_to_grid(x, 23, -126, 127)
    if isinstance(r, str):
        raise OverflowError("binary32 overflow")
    return r


def bf16(x: F):
    """Round to BF16 (8-bit significand, binary32's exponent range)."""
    return round_to_grid(x, 7, -126, 127)


def bf16_bits(v) -> int:
    """BF16 bit pattern of an exactly representable value (or 'inf'/'-inf')."""
    if v == "inf":
        return 0x7F80
    if v == "-inf":
        return 0xFF80
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    if a == 0:
        return sign
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    elif F(2) ** (e + 1) <= a:
        e += 1
    if e < -126:  # subnormal: a = m * 2^-133
        m = a / F(2) ** -133
        assert m.denominator == 1 and 0 < m < 128
        return sign | int(m)
    m = a / F(2) ** e - 1
    frac = m * 128
    assert frac.denominator == 1
    return sign | ((e + 127) << 7) | int(frac)


def bits_to_value(b: int) -> F:
    """Exact value of a finite BF16 bit pattern."""
    sign = -1 if b & 0x8000 else 1
    ex = (b >> 7) & 0xFF
    m = b & 0x7F
    assert ex != 0xFF
    if ex == 0:
        return sign * F(m) * F(2) ** -133
    return sign * (1 + F(m, 128)) * F(2) ** (ex - 127)


def f32_value(x: float) -> F:
    return F(x)  # a Python float holding a binary32 value converts exactly


# ---- E4M3 (OCP): 3 fraction bits, exponent bias 7, max finite 448, 0x7F NaN
def e4m3_values():
    """All 126 non-negative finite E4M3 values with their codes (0x00..0x7E)."""
    out = []
    for code in range(0x7F):
        e = code >> 3
        m = code & 7
        if e == 0:
            v = F(m) * F(2) ** -9
        else:
            v = (1 + F(m, 8)) * F(2) ** (e - 7)
        out.append((code, v))
    return out


_E4M3 = e4m3_values()


def e4m3_nearest(y: F) -> int:
    """Brute force over all codes: nearest value, ties to the even code, saturate to 448,
    sign of zero from the sign of y (negative y that rounds to zero -> 0x80)."""
    sign = 0x80 if y < 0 else 0
    a = abs(y)
    best = None
    for code, v in _E4M3:
        d = abs(v - a)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return sign | best[1]


def e8m0_up(v: F) -> int:
    """Smallest b in [0, 254] with 2^(b-127) >= v (round toward +inf, saturate)."""
    for b in range(255):
        if F(2) ** (b - 127) >= v:
            return b
    return 254


# ---- the codec steps, in exact arithmetic plus explicit roundings
def quant_block_i8(vals):
    """vals: exact binary32 values of one 128-value block -> (q list, scale)."""
    amax = max(abs(v) for v in vals)
    s = f32(amax / 127)
    q = []
    for v in vals:
        if s == 0:
            q.append(0)
            continue
        t = f32(v / s)
        r = _round_half_even(t)
        q.append(max(-127, min(127, r)))
    return q, s


def bf16_bits_signed(x: F, negative: bool) -> int:
    """BF16 bit pattern of round(x), with the sign of a zero result taken from
    `negative` (IEEE rounding keeps the sign of a product that rounds to zero)."""
    r = bf16(x)
    if r == 0:
        return 0x8000 if negative else 0x0000
    return bf16_bits(r)


def dequant_i8(q: int, s: F) -> int:
    """Materialization: binary32 product, then BF16; q < 0 gives a negative zero when
    the product rounds to zero (s >= 0 always)."""
    p = f32(q * s)
    return bf16_bits_signed(p, q < 0 and s != 0)


# ---- MX wire reductions, with the sign of zero tracked (binary32 values as
# (exact value, is negative zero) pairs)
def f32_add_signed(a, b):
    """binary32 a + b (round to nearest even). A zero sum is -0 only when both
    operands are -0; a nonzero exact sum of two binary32 values never rounds to 0."""
    v = f32(a[0] + b[0])
    neg0 = v == 0 and a[0] == 0 and b[0] == 0 and a[1] and b[1]
    return v, neg0


def mx_element(code: int, e: int):
    """decode(code) * 2^(e-127) as (exact value, is negative zero)."""
    mag = dict(_E4M3)[code & 0x7F] * F(2) ** (e - 127)
    neg = bool(code & 0x80)
    return (-mag if neg else mag), (neg and mag == 0)


def quant_group_mx(vals):
    """vals: 32 (exact binary32 value, is negative zero) pairs -> (codes, E8M0 byte)."""
    amax = max(abs(v) for v, _ in vals)
    e = 127 if amax == 0 else e8m0_up(f32(amax / 448))
    codes = []
    for v, neg0 in vals:
        c = e4m3_nearest(v * F(2) ** (127 - e))
        if v == 0 and neg0:
            c = 0x80
        codes.append(c)
    return codes, e


def dequant_mx(code: int, e: int) -> int:
    """BF16 bits of decode(code) * 2^(e-127) (exact product, one rounding)."""
    v, _ = mx_element(code, e)
    return bf16_bits_signed(v, bool(code & 0x80))


# ---- legacy E4M3 codec (reading R14) and FP16 inputs
def quant_block_e4m3(vals):
    """vals: 128 (exact binary32 value, is negative zero) pairs -> (codes, scale)."""
    amax = max(abs(v) for v, _ in vals)
    s = f32(amax / 448)
    codes = []
    for v, neg0 in vals:
        if s == 0:
            codes.append(0)
            continue
        t = f32(v / s)
        c = e4m3_nearest(t)
        if t == 0 and (neg0 or v < 0):
            c = 0x80
        codes.append(c)
    return codes, s


def dequant_e4m3(code: int, s: F) -> int:
    """BF16 bits of fl(decode(code) * s), then BF16 (two roundings)."""
    mag = dict(_E4M3)[code & 0x7F]
    neg = bool(code & 0x80)
    p = f32((-mag if neg else mag) * s)
    return bf16_bits_signed(p, neg and s != 0)


def f16_value(bits: int) -> F:
    """Exact value of an IEEE binary16 bit pattern, from its definition."""
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    if e == 0:
        return sign * F(f) * F(2) ** -24
    return sign * (1 + F(f, 1024)) * F(2) ** (e - 15)
