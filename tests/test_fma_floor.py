"""The page's floor-invisibility claim for the quantize rule, checked.

"Verification -- why you can trust the numbers", section "Hardware ground
truth (RDNA2 ISA audit)", claims that contracting x*inv + 0.5 into one fused
multiply-add (one rounding instead of two) can change the last bit of the sum
at binade edges but never the floor -- the int8 value.

On the exact-rational referee the first half holds (anomalies exist) but the
second fails in two narrow bands, both where the sum crosses an integer below
the binade edge at 1:
  * p = x*inv just below -1/2: two roundings give RN(p) = -1/2, a sum of
    exactly 0 and q = 0; the fused schedule keeps the negative residue
    p + 1/2 and floors it to q = -1;
  * p just below +1/2: RN(p) = 1/2 - 2^-25, and RN(p) + 1/2 = 1 - 2^-25 is a
    tie that goes to the even neighbour 1.0, so q = 1; the fused sum rounds
    to 1 - 2^-24 and q = 0.
The sweeps below find no other place where the floors part.  The oracle (and
the CUDA kernels) therefore fix the two-rounding schedule rather than lean on
the claim.
"""
import numpy as np

import referee as R

F32 = R.BINARY32


def fused_u(x_bits: int, inv_bits: int) -> int:
    """RN(x*inv + 1/2) with the product kept exact (one rounding)."""
    a, b = R.decode(x_bits, F32), R.decode(inv_bits, F32)
    sign = a.sign ^ b.sign
    num = a.mant * b.mant
    e = a.exp + b.exp                     # value = (-1)^sign num 2^e
    # + 1/2 = 2^(e) * 2^(-1-e)
    if e <= -1:
        half = 1 << (-1 - e)
        tot = (-num if sign else num) + half
        return R.round_rational(1 if tot < 0 else 0, abs(tot), 1 << -e, F32) if tot else 0
    tot = (-num if sign else num) * (1 << (e + 1)) + 1
    return R.round_rational(1 if tot < 0 else 0, abs(tot), 2, F32) if tot else 0


def sweep(seed: int, n_inv: int = 60):
    rng = np.random.default_rng(seed)
    invs = []
    for m in (10.0 ** rng.uniform(-7, 30, n_inv)).astype(np.float32):
        _, inv = R.ref_scale(int(np.array([m], np.float32).view(np.uint32)[0]))
        invs.append(inv)
    cases = []
    for inv in invs:
        invf = float(np.array([inv], np.uint32).view(np.float32)[0])
        targets = [k + 0.5 for k in range(-127, 127, 5)]
        targets += [2.0 ** p for p in range(-3, 8)] + [-(2.0 ** p) for p in range(-3, 8)]
        targets += [2.0 ** p - 0.5 for p in range(0, 8)] + [0.25, -0.25, 1e-3, -1e-3]
        for t in targets:
            x0 = np.float32(t / invf)
            xb = int(np.array([x0], np.float32).view(np.uint32)[0])
            for d in range(-6, 7):
                cases.append((xb + d, inv))
    return cases


def product(x: int, inv: int):
    return R.decode(x, F32).fraction() * R.decode(inv, F32).fraction()


def near_half_band(x: int, inv: int) -> bool:
    """True when the exact product is within 2^-23 below -1/2 or +1/2."""
    from fractions import Fraction
    p = product(x, inv)
    eps = Fraction(1, 2 ** 23)
    return any(h - eps <= p < h for h in (Fraction(-1, 2), Fraction(1, 2)))


def test_fma_floor_claim_on_referee():
    anomalies = 0
    survivors = 0
    total = 0
    for x, inv in sweep(0):
        if R.decode(x, F32).kind != "fin":
            continue
        two = R.add(R.mul(x, inv, F32), R.F32_HALF, F32)
        one = fused_u(x, inv)
        total += 1
        if two != one:
            anomalies += 1
            if R.floor_value(two, F32) != R.floor_value(one, F32):
                survivors += 1
                assert near_half_band(x, inv), (hex(x), hex(inv))
    print(f"{anomalies} last-bit anomalies in {total} cases; {survivors} reach the floor, "
          "all just below p = -1/2 or p = +1/2")
    assert anomalies > 0       # first half of the claim: anomalies exist


def test_floor_claim_counterexamples():
    """Concrete inputs where the two schedules give different int8 values."""
    # p just below -1/2: q = 0 with two roundings, -1 fused
    x, inv = 0xC071CC91, 0x3E078479
    two = R.add(R.mul(x, inv, F32), R.F32_HALF, F32)
    assert R.floor_value(two, F32) == 0 and R.floor_value(fused_u(x, inv), F32) == -1
    # p just below +1/2: q = 1 with two roundings, 0 fused
    x, inv = 0x325DECD6, 0x4C13A744
    two = R.add(R.mul(x, inv, F32), R.F32_HALF, F32)
    assert R.floor_value(two, F32) == 1 and R.floor_value(fused_u(x, inv), F32) == 0


def test_floor_disagreements_only_near_plus_minus_half_dense():
    """Dense scan around every half-integer target k + 1/2 in [-127, 127)."""
    rng = np.random.default_rng(5)
    seen = set()
    for _ in range(12):
        m = np.float32(10.0 ** rng.uniform(-6, 20))
        _, inv = R.ref_scale(int(np.array([m], np.float32).view(np.uint32)[0]))
        invf = float(np.array([inv], np.uint32).view(np.float32)[0])
        for k in range(-127, 127):
            xb = int(np.array([np.float32((k + 0.5) / invf)], np.float32).view(np.uint32)[0])
            for d in range(-5, 6):
                x = xb + d
                two = R.add(R.mul(x, inv, F32), R.F32_HALF, F32)
                one = fused_u(x, inv)
                if R.floor_value(two, F32) != R.floor_value(one, F32):
                    assert near_half_band(x, inv)
                    seen.add(k)
    assert seen <= {-1, 0}


def test_oracle_follows_two_roundings(orc):
    cases = sweep(1, 25)
    xs = np.array([c[0] for c in cases], np.uint32).view(np.float32)
    invs = np.array([c[1] for c in cases], np.uint32).view(np.float32)
    for x, inv, (xb, ib) in zip(xs, invs, cases):
        if not np.isfinite(x):
            continue
        q = orc.quantize_value(float(x), float(inv))
        two = R.add(R.mul(xb, ib, F32), R.F32_HALF, F32)
        assert q == R.floor_value(two, F32)
        if not near_half_band(xb, ib):
            assert q == R.floor_value(fused_u(xb, ib), F32)
    # on the counterexamples the oracle takes the two-rounding values
    for xb, ib, want in ((0xC071CC91, 0x3E078479, 0), (0x325DECD6, 0x4C13A744, 1)):
        cx = np.array([xb, ib], np.uint32).view(np.float32)
        assert orc.quantize_value(float(cx[0]), float(cx[1])) == want
