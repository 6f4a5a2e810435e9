"""Inputs on which plausible variants of the unit's rules give different
bytes from the rules themselves ("gate the gate").

"Verification -- why you can trust the numbers", section "Layer 1: exact init
gates": a gate is only meaningful if the input it uses makes the old or wrong
specification fail.  Each case below is found by a seeded search on the
exact-rational referee and carries the spec's answer and the variant's
different answer; the search never consults the oracle or the GPU.

Quantize cases are rows (1 x K, K >= 2) whose int8 values or scale differ
under the variant.  Epilogue cases are (s, a, b) triples.
"""
from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction
from functools import lru_cache

import numpy as np

import referee as R

F32, F64 = R.BINARY32, R.BINARY64


def b2f(b: int) -> np.float32:
    return np.array([b], np.uint32).view(np.float32)[0]


def f2b(x) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


# ---- the variants (each a plausible wrong reading) ----------------------
def inv_alpha(m: int) -> int:
    return R.ref_scale(m)[1]


def inv_beta(m: int) -> int:
    """inv = f32(1 / s64): the reciprocal of the unrounded f64 scale."""
    s64 = R.div(R.convert(m, F32, F64), R.F64_127, F64)
    if R.lt(s64, R.F64_1EM8, F64):
        s64 = R.F64_1EM8
    return R.convert(R.div(R.F64_ONE, s64, F64), F64, F32)


def inv_gamma(m: int) -> int:
    """inv = f32(127 / f64(m))."""
    m64 = R.convert(m, F32, F64)
    s64 = R.div(m64, R.F64_127, F64)
    if R.lt(s64, R.F64_1EM8, F64):
        return inv_alpha(m)
    return R.convert(R.div(R.F64_127, m64, F64), F64, F32)


def q_rne(x: int, inv: int) -> int:
    """Round half to even instead of floor(t + 1/2)."""
    t = R.decode(R.mul(x, inv, F32), F32).fraction()
    fl = t.numerator // t.denominator
    r = t - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def q_fused(x: int, inv: int) -> int:
    """One rounding: floor(RN(x*inv + 1/2))."""
    p = R.decode(x, F32).fraction() * R.decode(inv, F32).fraction() + Fraction(1, 2)
    if p == 0:
        return 0
    u = R.from_fraction(p, F32)
    return R.floor_value(u, F32)


def q_f64(x: int, inv: int) -> int:
    """The quantize in f64 (a JS number): floor(x*inv + 1/2) with f64 ops."""
    x64, i64 = R.convert(x, F32, F64), R.convert(inv, F32, F64)
    t = R.mul(x64, i64, F64)
    u = R.add(t, R.convert(R.F32_HALF, F32, F64), F64)
    return R.floor_value(u, F64)


def epi_round_once(s, a, b):
    return R.ref_epi_round_once(s, a, b)


def epi_swapped(s, a, b):
    return R.mul(R.mul(R.from_int(s, F32), b, F32), a, F32)


@dataclass
class RowCase:
    name: str
    row: np.ndarray          # float32 row (quantized alone)
    spec_q: list             # spec int8 values
    spec_scale: int          # spec scale bits


@dataclass
class EpiCase:
    name: str
    s: int
    a: int
    b: int
    spec: int
    variant: int


def _row_case(name, row):
    rb = [f2b(v) for v in row]
    sc, inv, q = R.ref_quantize_vector(rb)
    return RowCase(name, np.asarray(row, np.float32), q, sc)


def _search_inv_variant(variant, seed):
    rng = np.random.default_rng(seed)
    while True:
        m = np.float32(10.0 ** rng.uniform(-4, 6))
        mb = f2b(m)
        ia, iv = inv_alpha(mb), variant(mb)
        if ia == iv:
            continue
        invf = float(b2f(ia))
        for k in range(126, 100, -1):
            xb0 = f2b(np.float32((k + 0.5) / invf))
            for d in range(-12, 13):
                xb = xb0 + d
                if R.lt(mb, xb & 0x7FFFFFFF, F32):
                    continue
                qa = R.ref_quantize(xb, ia)
                qv = R.ref_quantize(xb, iv)
                if qa != qv:
                    return [m, b2f(xb)]


def _search_schedule(variant, seed, targets):
    rng = np.random.default_rng(seed)
    while True:
        m = np.float32(10.0 ** rng.uniform(-4, 6))
        mb = f2b(m)
        inv = inv_alpha(mb)
        invf = float(b2f(inv))
        for t in targets:
            xb0 = f2b(np.float32(t / invf))
            for d in range(-8, 9):
                xb = xb0 + d
                if R.lt(mb, xb & 0x7FFFFFFF, F32):
                    continue
                if R.ref_quantize(xb, inv) != variant(xb, inv):
                    return [m, b2f(xb)]


@lru_cache(maxsize=None)
def row_cases() -> list[RowCase]:
    cases = []
    # round-half-to-even instead of floor(x*inv + 1/2): unit scale, 2.5 -> 3
    cases.append(_row_case("rne_vs_half_up", [127.0, 2.5, -2.5, 0.5, -0.5, 4.5]))
    cases.append(_row_case("inv_beta", _search_inv_variant(inv_beta, 1)))
    cases.append(_row_case("inv_gamma", _search_inv_variant(inv_gamma, 2)))
    cases.append(_row_case("fused_minus_half", _search_schedule(q_fused, 3, [-0.5])))
    cases.append(_row_case("fused_plus_half", _search_schedule(q_fused, 4, [0.5])))
    cases.append(_row_case("f64_quantize", _search_schedule(q_f64, 5, [100.5, -60.5, 7.5])))
    # no 1e-8 floor: a 1e-30 row would quantize to +-127 instead of 0
    cases.append(_row_case("no_scale_floor", [1e-30, -5e-31, 2.5e-31]))
    # the zero-scale rule of the neighbouring weight-only scheme: scale 0
    cases.append(_row_case("zero_row_scale", [0.0, -0.0, 0.0]))
    return cases


def variant_of(case: RowCase):
    """(variant q list, variant scale bits) for a row case."""
    rb = [f2b(v) for v in case.row]
    m = R.ref_absmax(rb)
    sc, inv = R.ref_scale(m)
    name = case.name
    if name == "rne_vs_half_up":
        return [q_rne(x, inv) for x in rb], sc
    if name == "inv_beta":
        iv = inv_beta(m)
        return [R.ref_quantize(x, iv) for x in rb], sc
    if name == "inv_gamma":
        iv = inv_gamma(m)
        return [R.ref_quantize(x, iv) for x in rb], sc
    if name.startswith("fused"):
        return [q_fused(x, inv) for x in rb], sc
    if name == "f64_quantize":
        return [q_f64(x, inv) for x in rb], sc
    if name == "no_scale_floor":
        s64 = R.div(R.convert(m, F32, F64), R.F64_127, F64)
        s32 = R.convert(s64, F64, F32)
        iv = R.convert(R.div(R.F64_ONE, R.convert(s32, F32, F64), F64), F64, F32)
        return [R.ref_quantize(x, iv) for x in rb], s32
    if name == "zero_row_scale":
        return [0 for _ in rb], 0
    raise KeyError(name)


@lru_cache(maxsize=None)
def epi_cases() -> list[EpiCase]:
    rng = np.random.default_rng(11)
    out = []
    for name, fn in (("round_once", epi_round_once), ("swapped_order", epi_swapped)):
        found = 0
        while found < 8:
            s = int(rng.integers(-2 ** 31, 2 ** 31))
            a = f2b(np.float32(10.0 ** rng.uniform(-10, 2)))
            b = f2b(np.float32(10.0 ** rng.uniform(-10, 2)))
            spec, var = R.ref_epi(s, a, b), fn(s, a, b)
            if spec != var:
                out.append(EpiCase(name, s, a, b, spec, var))
                found += 1
    # the int->float conversion's tie: 2^24 + 1 must round to 2^24
    s, a, b = 2 ** 24 + 1, f2b(np.float32(1.0)), f2b(np.float32(1.0))
    out.append(EpiCase("int_to_float_tie", s, a, b, R.ref_epi(s, a, b),
                       R.from_int(2 ** 24 + 2, F32)))
    return out
