"""Pins of the oracle's whole unit: quantize -> exact int32 contraction ->
epilogue (+ReLU).

Rule: "Verification -- why you can trust the numbers", section "The verified
INT8 units" (steps 1-3) and section "Layer 5: properties and mutation scores"
(relations: row permutation, zero row, batch decomposition, single-cell
sensitivity; absolutes: fused ReLU never negative, unit scales give the exact
integer dot product).  Pins: big-integer brute force with the exact-rational
referee on 64 tiny shapes, numpy's int64 matmul, the properties.
"""
import numpy as np
import pytest

import referee as R
from verifiable_quantize_rows_gb300 import inputs

F32 = R.BINARY32


def u32(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def brute_force(A, B, relu):
    """Everything from the definitions: referee quantize per row/column,
    Python big-integer dot products, referee epilogue."""
    M, K = A.shape
    N = B.shape[1]
    Ab, Bb = u32(A), u32(B)
    ra = [R.ref_quantize_vector([int(x) for x in Ab[i]]) for i in range(M)]
    rb = [R.ref_quantize_vector([int(x) for x in Bb[:, j]]) for j in range(N)]
    C = np.zeros((M, N), np.uint32)
    S = np.zeros((M, N), np.int64)
    for i in range(M):
        for j in range(N):
            s = sum(qa * qb for qa, qb in zip(ra[i][2], rb[j][2]))
            S[i, j] = s
            c = R.ref_epi(s, ra[i][0], rb[j][0])
            C[i, j] = R.ref_relu(c) if relu else c
    return C, S


@pytest.mark.parametrize("idx", range(64))
def test_bruteforce_tiny_shapes(orc, idx):
    M, N, K, seed = inputs.tiny_shapes()[idx]
    A = inputs.normal((M, K), 1.0, seed).numpy()
    B = inputs.normal((K, N), 1.0, seed + 50_000).numpy()
    relu = bool(idx % 2)
    C, S, st = orc.bsgemm_i8(A, B, relu=relu, want_s=True)
    assert st == 0
    Cr, Sr = brute_force(A, B, relu)
    np.testing.assert_array_equal(S.astype(np.int64), Sr)
    np.testing.assert_array_equal(u32(C), Cr)


def test_bruteforce_adversarial_block(orc):
    A = inputs.adversarial(19, 23, 31).numpy()
    B = inputs.adversarial(17, 23, 32, along_rows=False).numpy()
    for relu in (False, True):
        C, S, st = orc.bsgemm_i8(A, B, relu=relu, want_s=True)
        assert st == 0
        Cr, Sr = brute_force(A, B, relu)
        np.testing.assert_array_equal(S.astype(np.int64), Sr)
        np.testing.assert_array_equal(u32(C), Cr)
    # the mix really reaches the edge cases
    C, _ = orc.bsgemm_i8(A, B)
    assert np.isinf(C).any() and (u32(C) == 0).any()


def test_contraction_is_textbook_integer_dot(orc):
    rng = np.random.default_rng(5)
    Aq = rng.integers(-127, 128, (70, 300)).astype(np.int8)
    Bq = rng.integers(-127, 128, (300, 90)).astype(np.int8)
    S, st = orc.gemm_s32(Aq, Bq)
    assert st == 0
    np.testing.assert_array_equal(S.astype(np.int64), Aq.astype(np.int64) @ Bq.astype(np.int64))


def test_int32_range_limit(orc):
    # K = 133144 saturated products fit int32; one more does not
    for K, ok in ((133144, True), (133145, False)):
        Aq = np.full((1, K), 127, np.int8)
        Bq = np.full((K, 1), 127, np.int8)
        S, st = orc.gemm_s32(Aq, Bq)
        assert (st == 0) == ok
        if ok:
            assert int(S[0, 0]) == 127 * 127 * K


def test_unit_scales_give_exact_integer_dot(orc):
    """Rows of A and columns of B whose absmax is 127 and whose values are
    integers quantize to themselves with scale 1, so C is the exact integer
    dot product (exactly representable while |dot| < 2^24)."""
    rng = np.random.default_rng(9)
    M, N, K = 33, 29, 700
    A = rng.integers(-127, 128, (M, K)).astype(np.float32)
    B = rng.integers(-127, 128, (K, N)).astype(np.float32)
    A[:, 0] = 127
    B[0, :] = -127
    C, st = orc.bsgemm_i8(A, B)
    assert st == 0
    exact = A.astype(np.int64) @ B.astype(np.int64)
    assert np.abs(exact).max() < 2 ** 24
    np.testing.assert_array_equal(C.astype(np.int64), exact)
    np.testing.assert_array_equal(C, exact.astype(np.float32))


def _case(seed, M=48, N=40, K=130):
    A = inputs.gpt2_activations(M, K, seed, outlier_frac=0.02).numpy()
    B = inputs.gpt2_weights(K, N, seed).numpy()
    return A, B


def test_relation_row_and_column_permutation(orc):
    A, B = _case(1)
    C, _ = orc.bsgemm_i8(A, B)
    rng = np.random.default_rng(1)
    pr, pc = rng.permutation(A.shape[0]), rng.permutation(B.shape[1])
    Cp, _ = orc.bsgemm_i8(A[pr], B[:, pc])
    np.testing.assert_array_equal(u32(Cp), u32(C[pr][:, pc]))


def test_relation_zero_row_gives_positive_zeros(orc):
    A, B = _case(2)
    A[5] = 0.0
    A[7] = -0.0
    for relu in (False, True):
        C, _ = orc.bsgemm_i8(A, B, relu=relu)
        assert not u32(C[5]).any() and not u32(C[7]).any()


def test_relation_batches_decompose(orc):
    A, B = _case(3)
    C, _ = orc.bsgemm_i8(A, B)
    parts = [orc.bsgemm_i8(A[a:b], B)[0] for a, b in ((0, 1), (1, 20), (20, 48))]
    np.testing.assert_array_equal(u32(np.concatenate(parts)), u32(C))
    cparts = [orc.bsgemm_i8(A, B[:, a:b])[0] for a, b in ((0, 13), (13, 40))]
    np.testing.assert_array_equal(u32(np.concatenate(cparts, axis=1)), u32(C))


def test_relation_single_cell_sensitivity(orc):
    A, B = _case(4)
    C, _ = orc.bsgemm_i8(A, B)
    A2 = A.copy()
    A2[9, 17] += 3.0      # changes row 9's values (and maybe its scale) only
    C2, _ = orc.bsgemm_i8(A2, B)
    diff = u32(C2) != u32(C)
    assert diff[9].any() and not np.delete(diff, 9, axis=0).any()
    B2 = B.copy()
    B2[11, 6] -= 1.0
    C3, _ = orc.bsgemm_i8(A, B2)
    diff = u32(C3) != u32(C)
    assert diff[:, 6].any() and not np.delete(diff, 6, axis=1).any()


def test_absolute_relu_never_negative(orc):
    A, B = _case(5)
    C, _ = orc.bsgemm_i8(A, B, relu=True)
    assert not (u32(C) >> 31).any()
    C0, _ = orc.bsgemm_i8(A, B, relu=False)
    assert (C0 < 0).any()


def test_cells_match_full(orc):
    A, B = _case(6, 64, 70, 300)
    for relu in (False, True):
        C, S, st = orc.bsgemm_i8(A, B, relu=relu, want_s=True)
        rng = np.random.default_rng(6)
        rows = rng.integers(0, 64, 200)
        cols = rng.integers(0, 70, 200)
        out, Sc, st2 = orc.bsgemm_cells(A, B, rows, cols, relu=relu)
        assert st == st2 == 0
        np.testing.assert_array_equal(u32(out), u32(C[rows, cols]))
        np.testing.assert_array_equal(Sc, S[rows, cols])
