"""Mutation score of the oracle's pins.

"Verification -- why you can trust the numbers", section "Layer 5": a checker
that has never rejected anything is decoration, so the checkers are scored
against planted bugs.  The page's external bug corpus is not used (it is not
available here); these are our own mutants, each a plausible mistake in the
oracle's C source (a dropped term, a wrong sign or index, a transposed
operand, a different rounding schedule).  Each is planted in a copy of the
oracle source, compiled, loaded, and run through a compact battery of the
pins; every mutant must be caught and the unmutated control must pass.
"""
import hashlib
import os
import shutil

import numpy as np
import pytest

import oracle
import referee as R
import gate_cases as G
from verifiable_quantize_rows_gb300 import inputs

SRC = os.path.join(os.path.dirname(oracle.__file__), "bsg_oracle.c")

MUTANTS = {
    "round_once_epilogue": [("float t = f * a;    /* RN */\n    float c = t * b;    /* RN */",
                             "float t = f;\n    float c = (float)((double)t * (double)a * (double)b);")],
    "epilogue_order_swapped": [("float t = f * a;", "float t = f * b;"),
                               ("float c = t * b;", "float c = t * a;")],
    "int_to_float_toward_zero": [("float f = (float)s; /* RN from int32 */",
                                  "float f = (float)s;\n    if (s > 0 && (double)f > (double)s) f = nextafterf(f, 0.0f);\n"
                                  "    if (s < 0 && (double)f < (double)s) f = nextafterf(f, 0.0f);")],
    "flush_subnormal_outputs": [("    float c = t * b;    /* RN */\n    return c;",
                                 "    float c = t * b;    /* RN */\n    if (fabsf(c) < 1.17549435e-38f) c = 0.0f * c;\n    return c;")],
    "quantize_round_half_even": [("float f = floorf(u);", "float f = nearbyintf(t);")],
    "quantize_fused_multiply_add": [("float u = t + 0.5f;  /* RN */", "float u = fmaf(x, inv, 0.5f);")],
    "quantize_in_f64": [("float t = x * inv;   /* RN */\n    float u = t + 0.5f;  /* RN */\n    float f = floorf(u);",
                         "double t = (double)x * (double)inv;\n    double u = t + 0.5;\n    float f = (float)floor(u);")],
    "inv_from_unrounded_scale": [("*inv = (float)(1.0 / (double)sf); /* R2 */", "*inv = (float)(1.0 / s);")],
    "inv_as_127_over_max": [("*inv = (float)(1.0 / (double)sf); /* R2 */",
                             "*inv = (s > 1e-8) ? (float)(127.0 / (double)m) : (float)(1.0 / (double)sf);")],
    "no_scale_floor": [("if (s < 1e-8) s = 1e-8;", "")],
    "divide_by_128": [("(double)m / 127.0", "(double)m / 128.0")],
    "signed_max_not_absmax": [("float a = fabsf(v); /* |-0| = +0 */", "float a = v;")],
    "nan_not_flagged": [("if (!isfinite(v)) finite = 0;", "if (isinf(v)) finite = 0;")],
    "absmax_skips_last": [("for (int64_t k = 0; k < n; ++k) {\n        float v = x[k * stride];",
                           "for (int64_t k = 0; k < n - 1; ++k) {\n        float v = x[k * stride];")],
    "dropped_k_tail": [("for (int64_t k = 0; k < K; ++k) {\n                int64_t a = Aq[i * K + k];",
                        "for (int64_t k = 0; k < K - 1; ++k) {\n                int64_t a = Aq[i * K + k];")],
    "subtracted_product": [("acc[j] += a * (int64_t)brow[j];", "acc[j] -= a * (int64_t)brow[j];")],
    "transposed_b_operand": [("acc[j] += a * (int64_t)brow[j];",
                              "acc[j] += a * (int64_t)Bq[(j * K + k) % (K * N)]; (void)brow;")],
    "int32_overflow_unchecked": [("if (acc[j] > INT32_MAX || acc[j] < INT32_MIN) local = ORC_ERR_RANGE;", "")],
    "scales_transposed": [("float c = orc_epi(S[i * N + j], sa[i], sb[j]);",
                           "float c = orc_epi(S[i * N + j], sa[j % (M ? M : 1)], sb[i % (N ? N : 1)]);")],
    "relu_keeps_negative_zero": [("return (c > 0.0f) ? c : 0.0f;", "return (c >= 0.0f) ? c : 0.0f;")],
    "relu_dropped": [("C[i * N + j] = relu ? orc_relu(c) : c;", "C[i * N + j] = c;")],
    "blake2s_rotation": [("    v[b] = rotr32(v[b] ^ v[c], 7);", "    v[b] = rotr32(v[b] ^ v[c], 8);")],
    "hash_last_node_flag_missing": [("                    l == nleaf - 1, cur + 32 * l);",
                                     "                    0, cur + 32 * l);")],
    "hash_node_depth_not_counted": [("                        (uint64_t)g, depth, 32, g == next - 1, nxt + 32 * g);",
                                     "                        (uint64_t)g, 1, 32, g == next - 1, nxt + 32 * g);")],
    "hash_fanin_2": [("#define ORC_FANIN 4", "#define ORC_FANIN 2")],
    "hash_leaf_128": [("#define ORC_LEAF_BYTES 256", "#define ORC_LEAF_BYTES 128")],
    "hash_column_major": [("uint8_t *p = bytes + 4 * (size_t)(i * N + j);",
                           "uint8_t *p = bytes + 4 * (size_t)(j * M + i);")],
    "splitmix_constant": [("0xbf58476d1ce4e5b9ull", "0xbf58476d1ce4e5b8ull")],
    "probe_b_stream_offset": [("orc_splitmix64(seed, (uint64_t)(M * K + e))",
                               "orc_splitmix64(seed, (uint64_t)(e + 1))")],
    "probe_value_offset": [("int32_t v = (int32_t)(z >> 40) - (1 << 23);",
                            "int32_t v = (int32_t)(z >> 40) - (1 << 22);")],
    "wquant_round_half_up": [("return lrint((double)w / (double)s);",
                              "return (long)floor((double)w / (double)s + 0.5);")],
    "wquant_divide_by_2_pow_b": [("float s = m / qmax;", "float s = m / (qmax + 1.0f);")],
    "wquant_pow2_rounds_down": [("return ldexpf(1.0f, e);        /* 2^e",
                                 "return ldexpf(1.0f, e - 1);    /* 2^e")],
    "wquant_zero_channel_floored": [("float s = m / qmax;", "float s = fmaxf(m / qmax, 1e-8f);")],
    "wquant_subnormal_scale_flushed": [("float s = m / qmax;",
                                        "float s = m / qmax;\n        if (s < 1.17549435e-38f) s = 0.0f;")],
    "int4_nibbles_swapped": [("P[k * ldp + i] = (uint8_t)(lo | (hi << 4));",
                              "P[k * ldp + i] = (uint8_t)(hi | (lo << 4));")],
    "wdequant_next_channel_scale": [("What[k * ldo + j] = (float)Q[k * ldq + j] * scale[j];",
                                     "What[k * ldo + j] = (float)Q[k * ldq + j] * scale[(j + 1) % N];")],
}


def _u32(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _tree_py(data: bytes) -> bytes:
    from test_hash import tree_hash_py
    return tree_hash_py(data)


def _splitmix_py(seed, i):
    mask = (1 << 64) - 1
    z = (seed + (i + 1) * 0x9E3779B97F4A7C15) & mask
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
    return z ^ (z >> 31)


# ---- the battery: each returns normally when its pin holds -------------
def pin_quantize_referee(o):
    rows = [inputs.normal((1, 40), 1.0, 3).numpy()[0],
            inputs.gpt2_activations(1, 64, 4, outlier_frac=0.05).numpy()[0],
            np.float32([1e-30, -3e-31, 5e-31]), np.float32([0.0, -0.0]),
            np.float32([5.0])]
    rows += [c.row for c in G.row_cases()]
    rows += [inputs._adversarial_vector(k, 30, inputs._gen(40 + i)).numpy()
             for i, k in enumerate(inputs.ADVERSARIAL_KINDS)]
    for row in rows:
        Q, sc, iv, st = o.quantize_rows(row[None, :])
        s, i, q = R.ref_quantize_vector([int(b) for b in _u32(row)])
        assert int(_u32(sc)[0]) == s and int(_u32(iv)[0]) == i
        assert list(Q[0].astype(int)) == q


def pin_epilogue_referee(o):
    rng = np.random.default_rng(0)
    M, N = 60, 60
    S = rng.integers(-2 ** 31, 2 ** 31, (M, N)).astype(np.int32)
    S[0, :40] = [2 ** 24 + j for j in range(-20, 20)]
    sa = (10.0 ** rng.uniform(-10, 2, M)).astype(np.float32)
    sb = (10.0 ** rng.uniform(-10, 2, N)).astype(np.float32)
    sb[:3] = np.array([1, 0x80000001, 5], np.uint32).view(np.float32)   # subnormals
    sa[:2] = np.float32([1e-30, -1e-30])
    C = _u32(o.epilogue(S, sa, sb, relu=False))
    for i in range(M):
        for j in range(N):
            assert int(C[i, j]) == R.ref_epi(int(S[i, j]), int(_u32(sa)[i]), int(_u32(sb)[j]))
    Cr = _u32(o.epilogue(S, sa, sb, relu=True))
    assert not (Cr >> 31).any()
    assert (Cr == np.where(C.view(np.float32) > 0, C, 0)).all()


def pin_bruteforce(o):
    from test_oracle_gemm import brute_force
    for M, N, K, seed in inputs.tiny_shapes(6) + [(3, 5, 40, 77)]:
        A = inputs.normal((M, K), 1.0, seed).numpy()
        B = inputs.normal((K, N), 1.0, seed + 50_000).numpy()
        C, S, st = o.bsgemm_i8(A, B, relu=False, want_s=True)
        Cr, Sr = brute_force(A, B, False)
        assert (S.astype(np.int64) == Sr).all() and (_u32(C) == Cr).all()
    A = inputs.adversarial(9, 12, 5).numpy()
    B = inputs.adversarial(7, 12, 6, along_rows=False).numpy()
    C, S, st = o.bsgemm_i8(A, B, relu=True, want_s=True)
    Cr, Sr = brute_force(A, B, True)
    assert (S.astype(np.int64) == Sr).all() and (_u32(C) == Cr).all()


def pin_unit_scales(o):
    rng = np.random.default_rng(9)
    A = rng.integers(-127, 128, (9, 50)).astype(np.float32)
    B = rng.integers(-127, 128, (50, 7)).astype(np.float32)
    A[:, 0] = 127
    B[0, :] = -127
    C, _ = o.bsgemm_i8(A, B)
    assert (C.astype(np.int64) == A.astype(np.int64) @ B.astype(np.int64)).all()


def pin_int32_range(o):
    K = 133145
    S, st = o.gemm_s32(np.full((1, K), 127, np.int8), np.full((K, 1), 127, np.int8))
    assert st != 0


def pin_nonfinite(o):
    # a NaN alone, and an Inf alone, flag the row, the column and the weight
    # channel that hold them (the boundary's rule: inputs must be finite, and
    # a non-finite one is reported in the status)
    for bad in (np.nan, np.inf):
        A = np.ones((2, 8), np.float32)
        A[1, 5] = bad
        assert o.quantize_rows(A)[3] == 5
        assert o.quantize_cols(np.ascontiguousarray(A.T))[3] == 5
        assert o.wquant_cols(np.ascontiguousarray(A.T), 8, False)[2] == 5
    assert o.quantize_rows(np.ones((2, 8), np.float32))[3] == 0


def pin_zero_row(o):
    A = inputs.normal((5, 30), 1.0, 1).numpy()
    A[2] = -0.0
    C, _ = o.bsgemm_i8(A, inputs.normal((30, 4), 1.0, 2).numpy())
    assert not _u32(C[2]).any()


def pin_hash(o):
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "blake2s_rfc7693.txt")):
        if line.strip() and not line.startswith("#"):
            msg, dig = line.split()
            assert o.blake2s(msg.encode()).hex() == dig
    data = np.random.default_rng(1).integers(0, 256, 70_000, dtype=np.uint8).tobytes()
    assert o.tree_hash(data) == _tree_py(data)
    Cm = np.random.default_rng(2).standard_normal((7, 5)).astype(np.float32)
    assert o.hash_f32(Cm) == _tree_py(Cm.astype("<f4").tobytes())


def pin_probe(o):
    for i in range(3):
        assert o.splitmix64(0, i) == _splitmix_py(0, i)
    A, B = o.probe_inputs(3, 4, 5, 6)
    for e in range(24):
        z = _splitmix_py(3, e)
        assert A.reshape(-1)[e] == np.float32(((z >> 40) - 2 ** 23) / 2 ** 23)
    for e in range(30):
        z = _splitmix_py(3, 24 + e)
        assert B.reshape(-1)[e] == np.float32(((z >> 40) - 2 ** 23) / 2 ** 23)


def pin_wquant(o):
    from fractions import Fraction
    from test_oracle_wquant import columns, frac, rne, bits
    for b, p in ((8, False), (4, True)):
        W = columns(13, 9, b)
        Q, s, _ = o.wquant_cols(W, b, p)
        qmax = 2 ** (b - 1) - 1
        What = o.wdequant_cols(Q, s)
        for j in range(W.shape[1]):
            m = max(abs(frac(w)) for w in W[:, j])
            sa = R.decode(R.from_fraction(m / qmax, F32), F32).fraction()
            want = sa
            if p and sa:
                want = Fraction(1)
                while want < sa:
                    want *= 2
                while want / 2 >= sa:
                    want /= 2
            assert frac(s[j]) == want
            for k in range(W.shape[0]):
                q = 0 if want == 0 else rne(frac(W[k, j]) / want)
                assert int(Q[k, j]) == q
                assert bits(What[k, j]) == R.from_fraction(q * want, F32)
    Q4, _, _ = o.wquant_cols(np.float32([[3.0], [1.25], [0.75], [-1.25]]), 4, True)
    assert [int(v) for v in Q4[:, 0]] == [6, 2, 2, -2]
    P = o.pack_int4(np.array([[1, -1, 7]], np.int8))
    assert P[0, 0] == 0xF1 and P[0, 1] == 0x07


F32 = R.BINARY32

BATTERY = [pin_quantize_referee, pin_epilogue_referee, pin_bruteforce, pin_unit_scales,
           pin_int32_range, pin_nonfinite, pin_zero_row, pin_hash, pin_probe, pin_wquant]


def run_battery(o):
    """Names of the pins that caught something (empty: all pins hold)."""
    caught = []
    for pin in BATTERY:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    return caught


def _build_variant(tmp_path, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    cpath = d / "bsg_oracle.c"
    cpath.write_text(src)
    return oracle.load(oracle.compile_oracle(str(cpath), str(d / "lib.so")))


def test_control_passes(tmp_path):
    o = _build_variant(tmp_path, "control", [])
    assert run_battery(o) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    o = _build_variant(tmp_path, name, MUTANTS[name])
    caught = run_battery(o)
    assert caught, f"mutant {name} survived every pin"
