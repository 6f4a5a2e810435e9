"""The kernels derive scale and inv with two IEEE f32 divides instead of the
f64 divides the definition uses ("Verification -- why you can trust the
numbers", section "The verified INT8 units": scales come from f64, which is
exactly rounded).  The argument that the two agree is in quantize.cu; here
it is checked on the host, independently of the GPU:

    scale = max(RN32(m / 127), RN32(RN64(1e-8)))     inv = RN32(1 / scale)

against the oracle's f64 formula, for every mantissa at a spread of
exponents (including all subnormals and the binades around the 1e-8 floor),
and against the exact-rational referee on a sample.  The GPU side is
``bsg_selftest_scales`` (test_gpu_units.py), which compares the two device
formulas over every finite non-negative float.
"""
import numpy as np
import pytest

import referee as R

FLOOR_BITS = 0x322BCC77


def f32_formula(m):
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        s = np.maximum(m / np.float32(127.0), np.uint32(FLOOR_BITS).view(np.float32))
        inv = np.float32(1.0) / s
    return s.astype(np.float32), inv.astype(np.float32)


def test_floor_constant_is_f32_of_f64_1e8():
    assert FLOOR_BITS == R.convert(R.F64_1EM8, R.BINARY64, R.BINARY32)
    assert np.float32(np.float64(1e-8)).view(np.uint32) == FLOOR_BITS


@pytest.mark.parametrize("biased_exp", [0, 1, 2, 50, 100, 104, 105, 106, 107, 108, 109, 110,
                                        126, 127, 128, 200, 253, 254])
def test_every_mantissa_at_exponent(orc, biased_exp):
    bits = (np.uint32(biased_exp) << np.uint32(23)) | np.arange(1 << 23, dtype=np.uint32)
    m = bits.view(np.float32)
    s_ref, i_ref = orc.scales_from_max(m)
    s, i = f32_formula(m)
    np.testing.assert_array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    np.testing.assert_array_equal(i.view(np.uint32), i_ref.view(np.uint32))


def test_floor_boundary_dense(orc):
    center = np.float32(127e-8).view(np.uint32)
    bits = np.arange(int(center) - 200_000, int(center) + 200_000, dtype=np.uint32)
    m = bits.view(np.float32)
    s_ref, i_ref = orc.scales_from_max(m)
    s, i = f32_formula(m)
    np.testing.assert_array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    np.testing.assert_array_equal(i.view(np.uint32), i_ref.view(np.uint32))


def test_random_full_range_vs_referee():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 0x7F800000, 3000, dtype=np.uint64).astype(np.uint32)
    m = bits.view(np.float32)
    s, i = f32_formula(m)
    for b, sv, iv in zip(bits, s.view(np.uint32), i.view(np.uint32)):
        rs, ri = R.ref_scale(int(b))
        assert (int(sv), int(iv)) == (rs, ri)
