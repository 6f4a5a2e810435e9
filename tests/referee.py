"""An IEEE-754 referee written from the standard's definitions, in exact
integer arithmetic.

It follows the method of "Verification -- why you can trust the numbers",
section "Layer 4: the referee -- an IEEE-754 oracle": binary32 (and binary64)
results are formed from the exact rational value of each operation and then
rounded to nearest, ties to even, with subnormals, signed zero and overflow to
infinity as IEEE 754-2019 sections 4.3.1, 6.3 and 7.4 define them.  No
hardware float operation is used to round anything: a value is a sign, an
integer numerator and an integer denominator; a float is its bit pattern.

This module pins the oracle; it is independent of the oracle's C code and of
the CUDA library.
"""
from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction


@dataclass(frozen=True)
class Fmt:
    bits: int     # storage width
    p: int        # precision, hidden bit included
    emin: int
    emax: int

    @property
    def bias(self) -> int:
        return self.emax

    @property
    def ebits(self) -> int:
        return self.bits - self.p


BINARY32 = Fmt(32, 24, -126, 127)
BINARY64 = Fmt(64, 53, -1022, 1023)


def _inf_bits(fmt: Fmt, sign: int) -> int:
    return (sign << (fmt.bits - 1)) | (((1 << fmt.ebits) - 1) << (fmt.p - 1))


def nan_bits(fmt: Fmt) -> int:
    return _inf_bits(fmt, 0) | (1 << (fmt.p - 2))


def round_rational(sign: int, num: int, den: int, fmt: Fmt) -> int:
    """Bits of the value (-1)^sign * num/den rounded to nearest, ties to even.

    num >= 0, den > 0.  A zero magnitude keeps the given sign.
    """
    assert num >= 0 and den > 0
    sbit = sign << (fmt.bits - 1)
    if num == 0:
        return sbit
    # e = floor(log2(num/den))
    e = num.bit_length() - den.bit_length()
    if e >= 0:
        if num < (den << e):
            e -= 1
    else:
        if (num << -e) < den:
            e -= 1
    e_eff = max(e, fmt.emin)
    qe = e_eff - (fmt.p - 1)          # exponent of one unit in the last place
    if qe <= 0:
        n2, d2 = num << -qe, den
    else:
        n2, d2 = num, den << qe
    N, r = divmod(n2, d2)
    twice = 2 * r
    if twice > d2 or (twice == d2 and (N & 1)):
        N += 1
    if N == 0:
        return sbit
    if N >= (1 << fmt.p):              # carried into the next binade (N == 2^p)
        N >>= 1
        qe += 1
    if N < (1 << (fmt.p - 1)):         # subnormal
        return sbit | N
    E = qe + fmt.p - 1
    if E > fmt.emax:
        return _inf_bits(fmt, sign)
    return sbit | ((E + fmt.bias) << (fmt.p - 1)) | (N - (1 << (fmt.p - 1)))


@dataclass(frozen=True)
class Val:
    """A decoded float: kind in {'fin', 'inf', 'nan'}; finite value is
    (-1)^sign * mant * 2^exp (exact)."""
    kind: str
    sign: int
    mant: int = 0
    exp: int = 0

    def fraction(self) -> Fraction:
        assert self.kind == "fin"
        v = Fraction(self.mant) * (Fraction(2) ** self.exp)
        return -v if self.sign else v


def decode(bits: int, fmt: Fmt) -> Val:
    sign = (bits >> (fmt.bits - 1)) & 1
    be = (bits >> (fmt.p - 1)) & ((1 << fmt.ebits) - 1)
    frac = bits & ((1 << (fmt.p - 1)) - 1)
    if be == (1 << fmt.ebits) - 1:
        return Val("nan" if frac else "inf", sign)
    if be == 0:
        return Val("fin", sign, frac, fmt.emin - (fmt.p - 1))
    return Val("fin", sign, frac | (1 << (fmt.p - 1)), be - fmt.bias - (fmt.p - 1))


def _round_dyadic(sign: int, mant: int, exp: int, fmt: Fmt) -> int:
    if exp >= 0:
        return round_rational(sign, mant << exp, 1, fmt)
    return round_rational(sign, mant, 1 << -exp, fmt)


def mul(x: int, y: int, fmt: Fmt) -> int:
    a, b = decode(x, fmt), decode(y, fmt)
    sign = a.sign ^ b.sign
    if a.kind == "nan" or b.kind == "nan":
        return nan_bits(fmt)
    if a.kind == "inf" or b.kind == "inf":
        other = b if a.kind == "inf" else a
        if other.kind == "fin" and other.mant == 0:
            return nan_bits(fmt)            # 0 * inf is invalid
        return _inf_bits(fmt, sign)
    return _round_dyadic(sign, a.mant * b.mant, a.exp + b.exp, fmt)


def add(x: int, y: int, fmt: Fmt) -> int:
    a, b = decode(x, fmt), decode(y, fmt)
    if a.kind == "nan" or b.kind == "nan":
        return nan_bits(fmt)
    if a.kind == "inf" or b.kind == "inf":
        if a.kind == "inf" and b.kind == "inf" and a.sign != b.sign:
            return nan_bits(fmt)
        return _inf_bits(fmt, a.sign if a.kind == "inf" else b.sign)
    e = min(a.exp, b.exp)
    na = a.mant << (a.exp - e)
    nb = b.mant << (b.exp - e)
    s = (-na if a.sign else na) + (-nb if b.sign else nb)
    if s == 0:
        # exact zero sum under round-to-nearest: -0 only if both are -0
        sign = 1 if (a.sign and b.sign) else 0
        return sign << (fmt.bits - 1)
    return _round_dyadic(1 if s < 0 else 0, abs(s), e, fmt)


def div(x: int, y: int, fmt: Fmt) -> int:
    a, b = decode(x, fmt), decode(y, fmt)
    assert a.kind == "fin" and b.kind == "fin" and b.mant != 0
    sign = a.sign ^ b.sign
    # (ma 2^ea) / (mb 2^eb)
    num, den = a.mant, b.mant
    d = a.exp - b.exp
    if d >= 0:
        num <<= d
    else:
        den <<= -d
    return round_rational(sign, num, den, fmt)


def from_int(n: int, fmt: Fmt) -> int:
    return round_rational(1 if n < 0 else 0, abs(n), 1, fmt)


def convert(bits: int, src: Fmt, dst: Fmt) -> int:
    v = decode(bits, src)
    if v.kind == "nan":
        return nan_bits(dst)
    if v.kind == "inf":
        return _inf_bits(dst, v.sign)
    return _round_dyadic(v.sign, v.mant, v.exp, dst)


def from_fraction(q: Fraction, fmt: Fmt, negative_zero: bool = False) -> int:
    if q == 0:
        return (1 << (fmt.bits - 1)) if negative_zero else 0
    return round_rational(1 if q < 0 else 0, abs(q.numerator), q.denominator, fmt)


def floor_value(bits: int, fmt: Fmt) -> int:
    v = decode(bits, fmt)
    assert v.kind == "fin"
    q = v.fraction()
    return q.numerator // q.denominator


def lt(x: int, y: int, fmt: Fmt) -> bool:
    """IEEE x < y for non-NaN x, y (so -0 < +0 is false)."""
    a, b = decode(x, fmt), decode(y, fmt)
    assert a.kind != "nan" and b.kind != "nan"

    def key(v):
        if v.kind == "inf":
            return Fraction(-1 if v.sign else 1) * 10 ** 400
        return v.fraction()
    return key(a) < key(b)


def is_nan(bits: int, fmt: Fmt) -> bool:
    return decode(bits, fmt).kind == "nan"


F32_HALF = from_fraction(Fraction(1, 2), BINARY32)
F32_ZERO = 0
F64_127 = from_int(127, BINARY64)
F64_ONE = from_int(1, BINARY64)
F64_1EM8 = from_fraction(Fraction(1, 10 ** 8), BINARY64)  # the f64 nearest 1e-8


# -------------------------------------------------------------------------
# The unit's arithmetic, restated on the referee (the page "Verification --
# why you can trust the numbers", section "The verified INT8 units", with
# readings R1-R5 of the oracle's header).
# -------------------------------------------------------------------------
def ref_abs(bits: int) -> int:
    return bits & 0x7FFFFFFF


def ref_absmax(row_bits) -> int:
    m = 0
    for b in row_bits:
        a = ref_abs(b)
        if lt(m, a, BINARY32):
            m = a
    return m


def ref_scale(m_bits: int) -> tuple[int, int]:
    """(scale, inv) bits from the absmax m: scale = f32(max(f64(m)/127, 1e-8)),
    inv = f32(1/f64(scale))."""
    m64 = convert(m_bits, BINARY32, BINARY64)
    s64 = div(m64, F64_127, BINARY64)
    if lt(s64, F64_1EM8, BINARY64):
        s64 = F64_1EM8
    scale = convert(s64, BINARY64, BINARY32)
    inv64 = div(F64_ONE, convert(scale, BINARY32, BINARY64), BINARY64)
    return scale, convert(inv64, BINARY64, BINARY32)


def ref_quantize(x_bits: int, inv_bits: int) -> int:
    t = mul(x_bits, inv_bits, BINARY32)
    u = add(t, F32_HALF, BINARY32)
    return floor_value(u, BINARY32)


def ref_epi(s: int, a_bits: int, b_bits: int) -> int:
    f = from_int(s, BINARY32)
    t = mul(f, a_bits, BINARY32)
    return mul(t, b_bits, BINARY32)


def ref_relu(c_bits: int) -> int:
    if is_nan(c_bits, BINARY32):
        return 0
    return c_bits if lt(F32_ZERO, c_bits, BINARY32) else 0


def ref_epi_round_once(s: int, a_bits: int, b_bits: int) -> int:
    """The older mirror the page's referee rejects: one rounding of the exact
    product s*a*b."""
    a, b = decode(a_bits, BINARY32), decode(b_bits, BINARY32)
    if a.kind != "fin" or b.kind != "fin":
        return ref_epi(s, a_bits, b_bits)
    sign = (1 if s < 0 else 0) ^ a.sign ^ b.sign
    return _round_dyadic(sign, abs(s) * a.mant * b.mant, a.exp + b.exp, BINARY32)


def ref_quantize_vector(row_bits) -> tuple[int, int, list[int]]:
    m = ref_absmax(row_bits)
    scale, inv = ref_scale(m)
    return scale, inv, [ref_quantize(b, inv) for b in row_bits]
