"""Pins of the oracle's presk weight storage (int8 / int4 codes, per-channel scales).

Rule: "Precision" manual (docs.presk-lang.org/presk_manual/precision), section
"Integer weights". Weights are stored with one scale per channel, over the
contracted axis:
- s = max|w| / (2^(b-1) - 1), rounded to f32;
- the "pow2" scheme rounds s up to a power of two, so that q*s is exact;
- an all-zero channel gets s = 0 and stores zeros;
- a stored weight means f32(q*s);
- the page's error rule: |w - w_hat| <= s/2 plus one f32 rounding of q*s.

The readings P1-P4 are listed in the oracle source. The pins below are
independent of it:
- exact rationals: the scale, and the nearest integer with ties to even;
- constructed ties;
- the page's error rule;
- pow2 exactness;
- the zero and underflow channels, and a channel of subnormal entries;
- the int4 nibble layout.
"""
from fractions import Fraction

import numpy as np
import pytest

import referee as R

F32 = R.BINARY32


def bits(x) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def frac(x) -> Fraction:
    return R.decode(bits(x), F32).fraction()


def rne(x: Fraction) -> int:
    """Nearest integer, ties to even (reading P1, from the definition)."""
    fl = x.numerator // x.denominator
    d = x - fl
    if d > Fraction(1, 2):
        return fl + 1
    if d < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def columns(K, N, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((K, N)) * scale).astype(np.float32)
    W[:, 0] = 0.0                                   # all-zero channel
    if N > 2:
        W[:, 1] = np.float32(2.0 ** -149)           # absmax/7 and /127 round to 0 (reading P2)
    if N > 3:
        # subnormal entries: a subnormal, non-zero scale (its reciprocal is
        # beyond binary32's range, so no product with it can give the codes)
        W[:, 2] = (rng.standard_normal(K) * 2.0 ** -130).astype(np.float32)
    return W


@pytest.mark.parametrize("bits_,pow2", [(8, False), (8, True), (4, False), (4, True)])
def test_scales_and_codes_against_exact_rationals(orc, bits_, pow2):
    W = columns(37, 23, bits_ + 10 * pow2)
    Q, s, st = orc.wquant_cols(W, bits_, pow2)
    assert st == 0
    qmax = 2 ** (bits_ - 1) - 1
    for j in range(W.shape[1]):
        m = max(abs(frac(w)) for w in W[:, j])
        s_abs = R.from_fraction(m / qmax, F32)          # m / qmax rounded to f32
        if pow2:
            sa = R.decode(s_abs, F32).fraction()
            if sa == 0:
                want = Fraction(0)
            else:
                want = Fraction(1)
                while want < sa:
                    want *= 2
                while want / 2 >= sa:
                    want /= 2
            assert frac(s[j]) == want, j
        else:
            assert bits(s[j]) == s_abs, j
        sj = frac(s[j])
        for k in range(W.shape[0]):
            q = 0 if sj == 0 else rne(frac(W[k, j]) / sj)
            assert int(Q[k, j]) == q, (j, k)
            assert abs(q) <= qmax


def test_ties_go_to_even(orc):
    # a channel whose pow2 scale is 1/2 and whose entries are odd quarters: w/s = k + 1/2
    col = np.array([3.0, 1.25, 0.75, -1.25, -0.75, 0.25, -0.25, 1.75], np.float32)
    W = col.reshape(-1, 1)
    Q, s, _ = orc.wquant_cols(W, 8, True)
    # m = 3 -> 3/127 rounded up to a power of two is 2^-5
    assert s[0] == np.float32(2.0 ** -5)
    Q4, s4, _ = orc.wquant_cols(W, 4, True)
    assert s4[0] == np.float32(0.5)                   # 3/7 -> 1/2
    want = [6, 2, 2, -2, -2, 0, 0, 4]                 # 2.5->2, 1.5->2, -2.5->-2, 0.5->0, 3.5->4
    assert [int(v) for v in Q4[:, 0]] == want


def test_zero_and_underflow_channels_store_zeros(orc):
    W = columns(9, 5, 1)
    for b in (8, 4):
        for p in (False, True):
            Q, s, _ = orc.wquant_cols(W, b, p)
            assert s[0] == 0 and s[1] == 0
            assert not Q[:, :2].any()


@pytest.mark.parametrize("bits_", [8, 4])
def test_error_rule_of_the_page(orc, bits_):
    W = columns(64, 40, 7, scale=3.0)
    Q, s, _ = orc.wquant_cols(W, bits_, False)
    What = orc.wdequant_cols(Q, s)
    for j in range(2, W.shape[1]):
        sj = frac(s[j])
        for k in range(W.shape[0]):
            w, wh = frac(W[k, j]), frac(What[k, j])
            q = int(Q[k, j])
            assert abs(w - q * sj) <= sj / 2                      # the rounding of w/s
            assert bits(What[k, j]) == R.from_fraction(q * sj, F32)  # f32(q*s), one rounding
            ulp = Fraction(2) ** (R.decode(bits(wh), F32).exp) if wh != 0 else 0
            assert abs(w - wh) <= sj / 2 + ulp


@pytest.mark.parametrize("bits_", [8, 4])
def test_pow2_products_are_exact(orc, bits_):
    W = columns(50, 30, 3, scale=0.7)
    Q, s, _ = orc.wquant_cols(W, bits_, True)
    What = orc.wdequant_cols(Q, s)
    for j in range(W.shape[1]):
        sj = frac(s[j])
        if sj:
            assert sj.numerator == 1 or sj.denominator == 1      # a power of two
        for k in range(W.shape[0]):
            assert frac(What[k, j]) == int(Q[k, j]) * sj


def test_pow2_ceil_closed_forms(orc):
    assert orc.pow2_ceil(3.0) == 4.0
    assert orc.pow2_ceil(4.0) == 4.0
    assert orc.pow2_ceil(0.0) == 0.0
    assert orc.pow2_ceil(float(np.float32(0.3))) == 0.5
    assert orc.pow2_ceil(2.0 ** -140) == 2.0 ** -140          # subnormal powers of two stay


def test_int4_nibble_layout(orc):
    Q = np.array([[1, -1, 7, -7, 0], [-8 + 1, 3, -2, 5, -3]], np.int8)
    P = orc.pack_int4(Q)
    assert P.shape == (2, 3)
    assert P[0, 0] == (1 | (0xF << 4))          # col 0 low nibble, col 1 (-1 = 0xF) high
    assert P[0, 1] == (7 | (0x9 << 4))          # -7 = 0x9
    assert P[0, 2] == 0                         # last odd column: high nibble zero
    lo = (P & 0x0F).astype(np.int16)
    hi = (P >> 4).astype(np.int16)
    lo = np.where(lo > 7, lo - 16, lo)
    hi = np.where(hi > 7, hi - 16, hi)
    back = np.stack([lo, hi], axis=2).reshape(2, 6)[:, :5]
    assert (back == Q).all()
