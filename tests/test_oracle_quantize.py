"""Pins of the oracle's quantize step (scale, inv, int8 values).

Rule: "Verification -- why you can trust the numbers", section "The verified
INT8 units", step 1 (scale = max|row|/127 floored at 1e-8; the scale is
derived in f64), and section "Hardware ground truth" (q = floor(x*inv+0.5)).
Pins: the exact-rational referee, closed forms for constructed ties and unit
scales, and the floor's boundary.
"""
import numpy as np
import pytest

import referee as R
from verifiable_quantize_rows_gb300 import inputs

F32 = R.BINARY32


def bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def f32(b: int) -> np.float32:
    return np.array([b], np.uint32).view(np.float32)[0]


def ref_rows(A):
    out_s, out_i, out_q = [], [], []
    for row in bits(A):
        s, i, q = R.ref_quantize_vector([int(b) for b in row])
        out_s.append(s), out_i.append(i), out_q.append(q)
    return np.array(out_s, np.uint32), np.array(out_i, np.uint32), np.array(out_q, np.int64)


@pytest.mark.parametrize("kind", ["normal", "gpt2", "wide_range"] + list(inputs.ADVERSARIAL_KINDS))
def test_quantize_rows_vs_referee(orc, kind):
    if kind == "normal":
        A = inputs.normal((24, 97), 1.0, 11).numpy()
    elif kind == "gpt2":
        A = inputs.gpt2_activations(16, 150, 12, outlier_frac=0.05).numpy()
    elif kind == "wide_range":
        rng = np.random.default_rng(13)
        A = (rng.uniform(-1, 1, (24, 61)) * 10.0 ** rng.integers(-35, 35, (24, 1))).astype(np.float32)
    else:
        A = np.stack([inputs._adversarial_vector(kind, 77, inputs._gen(100 + r)).numpy()
                      for r in range(12)])
    Q, sc, iv, st = orc.quantize_rows(A)
    assert st == 0
    rs, ri, rq = ref_rows(A)
    np.testing.assert_array_equal(bits(sc), rs)
    np.testing.assert_array_equal(bits(iv), ri)
    np.testing.assert_array_equal(Q.astype(np.int64), rq)
    assert Q.min() >= -127 and Q.max() <= 127


def test_quantize_cols_is_rows_of_transpose(orc):
    B = inputs.adversarial(40, 33, 21, along_rows=False).numpy()  # 33 x 40, kinds on columns
    Qc, sc, ic, st = orc.quantize_cols(B)
    Qr, sr, ir, st2 = orc.quantize_rows(np.ascontiguousarray(B.T))
    assert st == st2 == 0
    np.testing.assert_array_equal(Qc, Qr.T)
    np.testing.assert_array_equal(bits(sc), bits(sr))
    np.testing.assert_array_equal(bits(ic), bits(ir))
    # and against the referee column by column
    for j in range(B.shape[1]):
        s, i, q = R.ref_quantize_vector([int(b) for b in bits(B[:, j])])
        assert int(bits(sc)[j]) == s and list(Qc[:, j].astype(int)) == q


@pytest.mark.parametrize("e", [-20, -7, -1, 0, 1, 5, 20])
def test_constructed_ties_closed_form(orc, e):
    """max = 127*2^e gives scale = 2^e and inv = 2^-e exactly, so x =
    (k + 1/2) 2^e has x*inv = k + 1/2 exactly and q = k + 1 (ties go up)."""
    k = np.arange(-127, 127, dtype=np.int64)
    row = ((k + 0.5) * 2.0 ** e).astype(np.float32)
    row = np.concatenate([row, np.float32([127 * 2.0 ** e, -127 * 2.0 ** e])])
    Q, sc, iv, st = orc.quantize_rows(row[None, :])
    assert st == 0
    assert sc[0] == np.float32(2.0 ** e) and iv[0] == np.float32(2.0 ** -e)
    np.testing.assert_array_equal(Q[0, :-2].astype(np.int64), k + 1)
    assert Q[0, -2] == 127 and Q[0, -1] == -127
    # -2.5 -> -2 and 2.5 -> 3: round half up, not half to even
    assert Q[0, list(k).index(-3)] == -2 and Q[0, list(k).index(2)] == 3


def test_unit_scale_closed_form(orc):
    """max|row| = 127: scale 1, inv 1, q = floor(x + 1/2) for exactly
    representable x (quarter steps stay exact)."""
    x = np.arange(-127 * 4, 127 * 4 + 1, dtype=np.float64) / 4.0
    row = x.astype(np.float32)
    Q, sc, iv, st = orc.quantize_rows(row[None, :])
    assert sc[0] == 1.0 and iv[0] == 1.0
    np.testing.assert_array_equal(Q[0].astype(np.int64), np.floor(x + 0.5).astype(np.int64))


def test_zero_negzero_subnormal_rows_floor(orc):
    floor32 = f32(R.convert(R.F64_1EM8, R.BINARY64, F32))
    inv_floor = f32(R.convert(R.div(R.F64_ONE, R.convert(int(bits([floor32])[0]), F32, R.BINARY64),
                                    R.BINARY64), R.BINARY64, F32))
    rows = np.stack([
        np.zeros(50, np.float32),
        np.full(50, -0.0, np.float32),
        np.array([1e-45 * (i % 7) for i in range(50)], np.float32),   # subnormals
        np.full(50, 1e-30, np.float32),
        np.linspace(-1.27e-6, 1.27e-6, 50).astype(np.float32),        # m/127 ~ 1e-8
    ])
    Q, sc, iv, st = orc.quantize_rows(rows)
    assert st == 0
    for r in range(4):
        assert sc[r] == floor32 and iv[r] == inv_floor
        assert not Q[r].any()
    # the floor's boundary: f32(max(f64(m)/127, 1e-8)) agrees with the referee
    s, i, q = R.ref_quantize_vector([int(b) for b in bits(rows[4])])
    assert int(bits(sc)[4]) == s and list(Q[4].astype(int)) == q


def test_floor_boundary_sweep(orc):
    """Around m = 127e-8 the floor switches on; R1's two orders agree."""
    center = np.float32(127e-8)
    b0 = int(bits([center])[0])
    for d in range(-300, 301):
        m = int(b0 + d)
        s_ref, i_ref = R.ref_scale(m)
        s, i = orc.scale_from_max(float(f32(m)))
        assert int(bits([s])[0]) == s_ref and int(bits([i])[0]) == i_ref
        # floor applied after rounding to f32 gives the same scale (RN is monotone)
        m64 = R.convert(m, F32, R.BINARY64)
        q32 = R.convert(R.div(m64, R.F64_127, R.BINARY64), R.BINARY64, F32)
        fl32 = R.convert(R.F64_1EM8, R.BINARY64, F32)
        alt = fl32 if R.lt(q32, fl32, F32) else q32
        assert alt == s_ref


def test_nonfinite_rows_flagged(orc):
    A = np.ones((3, 8), np.float32)
    A[1, 3] = np.inf
    A[2, 0] = np.nan
    _, _, _, st = orc.quantize_rows(A)
    assert st == 5
    _, _, _, st = orc.quantize_rows(np.ones((2, 8), np.float32))
    assert st == 0
