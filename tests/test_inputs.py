"""The seeded input recipe: each adversarial kind has the property it is named
for, generation is reproducible, and the column form is the transpose of the
row form.  (The workloads' claims about what they exercise -- exact ties, the
1e-8 floor, subnormals, overflow -- rest on these properties.)"""
import numpy as np
import pytest

from verifiable_quantize_rows_gb300 import inputs

KINDS = inputs.ADVERSARIAL_KINDS


def vec(kind, n, seed):
    return inputs._adversarial_vector(kind, n, inputs._gen(seed)).numpy()


def u32(v):
    return np.ascontiguousarray(v, np.float32).view(np.uint32)


@pytest.mark.parametrize("n", [1, 7, 77, 300])
@pytest.mark.parametrize("seed", [0, 5, 123])
def test_each_kind_has_its_property(n, seed):
    v = vec("zero", n, seed)
    assert (u32(v) == 0).all()
    v = vec("neg_zero", n, seed)
    assert (u32(v) == 0x80000000).all()

    v = vec("ties", n, seed).astype(np.float64)
    m = np.abs(v).max()
    e = np.log2(m / 127.0)
    assert e == np.round(e)                       # max = 127 * 2^e exactly
    y = v / 2.0 ** e                              # exact: a power-of-two scale
    others = np.abs(y) != 127.0
    assert ((y[others] - 0.5) == np.round(y[others] - 0.5)).all()  # (k + 1/2) 2^e
    assert (np.abs(y[others]) < 127.0).all()

    bits = u32(vec("subnormal", n, seed)) & 0x7FFFFFFF
    assert ((bits > 0) & (bits < 0x00800000)).all()

    v = vec("subnormal_mix", n, seed)
    b = u32(v) & 0x7FFFFFFF
    sub = (b > 0) & (b < 0x00800000)
    assert (sub | (np.abs(v) < 1.0)).all()

    v = vec("huge", n, seed)
    assert (np.abs(v) <= 1e30).all() and np.abs(v).max() > 0
    v = vec("tiny", n, seed)
    assert (np.abs(v) <= 1e-30).all()             # max / 127 far below the 1e-8 floor

    v = vec("neg_max", n, seed)
    i = int(np.argmax(np.abs(v)))
    assert v[i] == -3.0 and (np.abs(np.delete(v, i)) <= 0.5).all()

    v = vec("spike", n, seed)
    i = int(np.argmax(np.abs(v)))
    assert v[i] == 1e4 and (np.abs(np.delete(v, i)) <= 1e-3).all()


def test_mixes_cover_every_kind_and_are_reproducible():
    rows, length = 40, 33
    A = inputs.adversarial(rows, length, 21).numpy()
    assert A.shape == (rows, length)
    assert np.array_equal(u32(A), u32(inputs.adversarial(rows, length, 21).numpy()))
    B = inputs.adversarial(rows, length, 21, along_rows=False).numpy()
    assert np.array_equal(u32(B), u32(A.T))
    # every kind is present: its signature is found in some row
    b = u32(A) & 0x7FFFFFFF
    found = {
        "zero": (u32(A) == 0).all(axis=1).any(),
        "neg_zero": (u32(A) == 0x80000000).all(axis=1).any(),
        "subnormal": ((b > 0) & (b < 0x00800000)).all(axis=1).any(),
        "huge": (np.abs(A).max(axis=1) > 1e20).any(),
        "tiny": ((np.abs(A).max(axis=1) < 1e-20) & (b.max(axis=1) > 0x00800000)).any(),
        "neg_max": (A.min(axis=1) == -3.0).any(),
        "spike": (A.max(axis=1) == 1e4).any(),
    }
    assert all(found.values()), found
    m = np.abs(A.astype(np.float64)).max(axis=1)
    ties = [r for r in range(rows) if m[r] > 0 and np.log2(m[r] / 127.0) == np.round(np.log2(m[r] / 127.0))]
    assert ties                                    # an exact-tie row
    assert len(set(KINDS)) == len(KINDS) == 9


def test_gpt2_activations_carry_outliers():
    A = inputs.gpt2_activations(512, 768, 3).numpy()
    base = inputs.normal((512, 768), 1.0, 3).numpy()
    changed = (A != base).mean()
    assert 0.0003 < changed < 0.003                # about 0.1 % of the entries scaled x20
