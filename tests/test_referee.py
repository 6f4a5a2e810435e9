"""Pins of the exact-rational IEEE-754 referee itself.

The referee rounds from the standard's definition in integer arithmetic; here
it is checked against (1) values the standard fixes by hand -- ties to even,
subnormal boundaries, overflow thresholds, signed zero -- and (2) the host
CPU's own IEEE binary32/binary64 hardware operations on random bit patterns.
"""
import numpy as np
import pytest
from fractions import Fraction

import referee as R

F32, F64 = R.BINARY32, R.BINARY64


def f2b(x) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def d2b(x) -> int:
    return int(np.array([x], np.float64).view(np.uint64)[0])


def test_hand_values_binary32():
    # 2^24 + 1 is halfway between 2^24 and 2^24 + 2: ties to even -> 2^24
    assert R.from_int(2 ** 24 + 1, F32) == 0x4B800000
    # 2^24 + 3 is halfway between 2^24 + 2 and 2^24 + 4 -> 2^24 + 4
    assert R.from_int(2 ** 24 + 3, F32) == 0x4B800002
    assert R.from_int(-(2 ** 24 + 3), F32) == 0xCB800002
    assert R.from_int(0, F32) == 0
    assert R.from_int(2 ** 31 - 1, F32) == 0x4F000000       # rounds up to 2^31
    assert R.from_int(-(2 ** 31), F32) == 0xCF000000
    # smallest subnormal, largest subnormal, smallest normal
    assert R.from_fraction(Fraction(1, 2 ** 149), F32) == 0x00000001
    assert R.from_fraction(Fraction(2 ** 23 - 1, 2 ** 149), F32) == 0x007FFFFF
    assert R.from_fraction(Fraction(1, 2 ** 126), F32) == 0x00800000
    # half the smallest subnormal is a tie between 0 and 2^-149: to even (0)
    assert R.from_fraction(Fraction(1, 2 ** 150), F32) == 0
    assert R.from_fraction(Fraction(3, 2 ** 151), F32) == 0x00000001
    # largest finite, and the overflow midpoint which rounds to infinity
    maxf = (2 ** 24 - 1) * 2 ** 104
    assert R.from_fraction(Fraction(maxf), F32) == 0x7F7FFFFF
    assert R.from_fraction(Fraction(2 ** 128 - 2 ** 103), F32) == 0x7F800000
    assert R.from_fraction(Fraction(2 ** 128 - 2 ** 103 - 1), F32) == 0x7F7FFFFF
    assert R.from_fraction(Fraction(1, 3), F32) == 0x3EAAAAAB


def test_signed_zero_rules():
    negz, posz = 0x80000000, 0
    one = f2b(1.0)
    assert R.mul(negz, one, F32) == negz
    assert R.mul(negz, f2b(-1.0), F32) == posz
    assert R.add(negz, negz, F32) == negz
    assert R.add(negz, posz, F32) == posz
    assert R.add(one, f2b(-1.0), F32) == posz
    # an underflowing product keeps its sign
    assert R.mul(f2b(-1e-30), f2b(1e-30), F32) == negz


def test_decode_roundtrip_exact():
    rng = np.random.default_rng(7)
    for b in rng.integers(0, 2 ** 32, 2000, dtype=np.uint64):
        b = int(b)
        v = R.decode(b, F32)
        if v.kind != "fin":
            continue
        assert R.from_fraction(v.fraction(), F32, negative_zero=bool(v.sign)) == b


@pytest.mark.parametrize("seed", [0, 1])
def test_against_host_ieee_binary32(seed):
    rng = np.random.default_rng(seed)
    n = 40000
    a = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    b = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    # half of the pairs get nearby exponents so sums cancel and round
    b[: n // 2] = (b[: n // 2] & 0x807FFFFF) | (a[: n // 2] & 0x7F800000)
    fa, fb = a.view(np.float32), b.view(np.float32)
    with np.errstate(all="ignore"):
        pm = (fa * fb).view(np.uint32)
        ps = (fa + fb).view(np.uint32)
    for i in range(n):
        x, y = int(a[i]), int(b[i])
        if R.is_nan(x, F32) or R.is_nan(y, F32):
            continue
        m, s = R.mul(x, y, F32), R.add(x, y, F32)
        assert (R.is_nan(m, F32) and np.isnan(pm[i:i + 1].view(np.float32)[0])) or m == int(pm[i])
        assert (R.is_nan(s, F32) and np.isnan(ps[i:i + 1].view(np.float32)[0])) or s == int(ps[i])


def test_against_host_ieee_binary64_div_and_convert():
    rng = np.random.default_rng(3)
    for _ in range(20000):
        with np.errstate(over="ignore"):
            m = np.float32(rng.uniform(0, 4) * 10.0 ** rng.integers(-40, 39))
        if not np.isfinite(m):
            continue
        m64 = d2b(np.float64(m))
        assert R.convert(f2b(m), F32, F64) == m64
        q = R.div(m64, R.F64_127, F64)
        assert q == d2b(np.float64(m) / np.float64(127.0))
        back = R.convert(q, F64, F32)
        assert back == f2b(np.float32(np.float64(m) / np.float64(127.0)))
        if np.float64(m) / 127.0 != 0:
            r = R.div(R.F64_ONE, q, F64)
            assert r == d2b(np.float64(1.0) / (np.float64(m) / np.float64(127.0)))


def test_f64_1e8_constant():
    assert R.F64_1EM8 == d2b(1e-8)
