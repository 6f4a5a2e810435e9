"""Pins of the oracle's epilogue epi(s,a,b) = f32(f32(f32(s)*a)*b) and ReLU.

Rule: "Verification -- why you can trust the numbers", section "The verified
INT8 units", step 3, and section "Layer 4: the referee" (500k+ checks, a
tie-to-even ladder around 2^24, subnormals, signed zero; the older round-once
mirror is rejected on a sizeable share of inputs).  Section "Layer 5": a
fused-ReLU output is never negative.
"""
import numpy as np

import referee as R

F32 = R.BINARY32


def epilogue_cases(seed: int, M: int = 1000, N: int = 520):
    """An M x N grid of (s, a, b): s per cell, a per row, b per column."""
    rng = np.random.default_rng(seed)
    # s: a quarter uniform int32, a quarter log-uniform magnitudes, half ladders
    n = M * N
    s = np.empty(n, np.int64)
    q = n // 4
    s[:q] = rng.integers(-2 ** 31, 2 ** 31, q)
    mag = rng.integers(0, 31, q)
    s[q:2 * q] = (rng.integers(0, 2 ** 31, q) >> (31 - mag)) * rng.choice([-1, 1], q)
    # tie-to-even ladders: +-(2^k + j), k = 24..30, j = -40..40
    ladder = np.array([sg * (2 ** k + j) for k in range(24, 31) for j in range(-40, 41)
                       for sg in (1, -1)], np.int64)
    s[2 * q:] = np.resize(ladder, n - 2 * q)
    s = np.clip(s, -2 ** 31, 2 ** 31 - 1)
    rng.shuffle(s)
    # a, b: random finite bit patterns (subnormals, +-0 included), realistic
    # positive scales, and exact powers of two
    def scales(k):
        out = np.empty(k, np.uint32)
        t = k // 3
        raw = rng.integers(0, 2 ** 32, t, dtype=np.uint64).astype(np.uint32)
        raw[(raw & 0x7F800000) == 0x7F800000] &= 0xBFFFFFFF   # no Inf/NaN
        raw[: t // 8] &= 0x807FFFFF                            # subnormals
        raw[t // 8: t // 8 + 4] = [0, 0x80000000, 1, 0x80000001]
        out[:t] = raw
        real = (10.0 ** rng.uniform(-8, 28, t) / 127.0).astype(np.float32)
        out[t:2 * t] = real.view(np.uint32)
        p2 = (2.0 ** rng.integers(-60, 60, k - 2 * t)).astype(np.float32)
        out[2 * t:] = p2.view(np.uint32)
        rng.shuffle(out)
        return out.view(np.float32)
    return s.reshape(M, N).astype(np.int32), scales(M), scales(N)


def test_epilogue_vs_referee_500k(orc):
    S, sa, sb = epilogue_cases(0)
    M, N = S.shape
    C = orc.epilogue(S, sa, sb, relu=False).view(np.uint32)
    sab, sbb = sa.view(np.uint32), sb.view(np.uint32)
    once_differs = 0
    checked = 0
    for i in range(M):
        a = int(sab[i])
        for j in range(N):
            s = int(S[i, j])
            r = R.ref_epi(s, a, int(sbb[j]))
            c = int(C[i, j])
            if R.is_nan(r, F32):
                assert R.is_nan(c, F32), (i, j)
            else:
                assert c == r, (i, j, s, hex(a), hex(int(sbb[j])), hex(c), hex(r))
            checked += 1
            if R.ref_epi_round_once(s, a, int(sbb[j])) != r and not R.is_nan(r, F32):
                once_differs += 1
    assert checked >= 500_000
    # the round-once mirror must be rejected on a non-trivial share of inputs
    rate = once_differs / checked
    print(f"round-once rejected on {100 * rate:.1f}% of {checked} inputs")
    assert rate > 0.05


def test_int_to_float_ladder_around_2p24(orc):
    one = np.float32(1.0)
    for k in range(24, 32):
        for j in range(-64, 65):
            for sg in (1, -1):
                s = sg * (2 ** k + j)
                if not (-2 ** 31 <= s < 2 ** 31):
                    continue
                c = orc.epi(s, one, one)
                assert int(np.array([c], np.float32).view(np.uint32)[0]) == R.from_int(s, F32)


def test_relu_never_negative_and_signed_zero(orc):
    S, sa, sb = epilogue_cases(1, 300, 300)
    C = orc.epilogue(S, sa, sb, relu=True)
    u = C.view(np.uint32)
    assert not (u >> 31).any()          # no sign bit anywhere, -0 included
    assert not np.isnan(C).any()
    assert np.array([orc.relu(-0.0)], np.float32).view(np.uint32)[0] == 0
    assert np.array([orc.relu(float("nan"))], np.float32).view(np.uint32)[0] == 0
    assert orc.relu(float("inf")) == float("inf")
    assert np.array([orc.relu(float("-inf"))], np.float32).view(np.uint32)[0] == 0
    # without ReLU, the same grid does produce -0 and negative values
    C0 = orc.epilogue(S, sa, sb, relu=False)
    assert (C0.view(np.uint32) == 0x80000000).any() and (C0 < 0).any()
    # ReLU is exactly max-with-+0 applied to the unfused output
    u0 = C0.view(np.uint32)
    expect = np.where((C0 > 0), u0, 0).astype(np.uint32)
    np.testing.assert_array_equal(u, expect)
