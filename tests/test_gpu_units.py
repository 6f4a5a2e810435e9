"""GPU parity of the unit's steps, one entry point at a time, through the C
ABI: quantize (rows, columns), the epilogue, the hash.  Every comparison is
bitwise against the CPU oracle on the same seeded inputs.
"""
import numpy as np
import pytest
import torch

import gate_cases as G
from gpu_util import assert_bits_equal, dev, host, u32
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu


def _matrix(kind, rows, cols, seed):
    if kind == "normal":
        return inputs.normal((rows, cols), 1.0, seed)
    if kind == "gpt2":
        return inputs.gpt2_activations(rows, cols, seed)
    if kind == "adversarial":
        return inputs.adversarial(rows, cols, seed)
    if kind == "uniform":
        return inputs.uniform((rows, cols), -1, 1, seed)
    raise KeyError(kind)


SHAPES = [(1, 1), (3, 5), (17, 13), (64, 768), (129, 1000), (300, 1024), (37, 1025),
          (8, 3072), (5, 5003), (1000, 33), (9, 16384), (2, 20000), (8200, 40), (16, 252),
          (2048, 96), (5000, 257)]


@pytest.mark.parametrize("kind", ["normal", "gpt2", "adversarial", "uniform"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_quantize_rows_bitwise(orc, kind, shape):
    X = _matrix(kind, *shape, seed=shape[0] * 7 + shape[1]).numpy()
    Q, sc, iv = bsg.quantize_rows(dev(X))
    Qo, sco, ivo, st = orc.quantize_rows(X)
    assert_bits_equal(host(Q), Qo, "Q")
    assert_bits_equal(host(sc), sco, "scale")
    assert_bits_equal(host(iv), ivo, "inv")


@pytest.mark.parametrize("kind", ["normal", "adversarial", "uniform"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_quantize_cols_bitwise(orc, kind, shape):
    # columns carry the adversarial kinds: build along rows, then transpose
    R, C = shape
    if kind == "adversarial":
        X = inputs.adversarial(C, R, seed=R + 3 * C, along_rows=False).numpy()
    else:
        X = _matrix(kind, R, C, seed=R * 5 + C).numpy()
    Q, sc, iv = bsg.quantize_cols(dev(X))
    Qo, sco, ivo, st = orc.quantize_cols(X)
    assert_bits_equal(host(Q), Qo, "Q")
    assert_bits_equal(host(sc), sco, "scale")
    assert_bits_equal(host(iv), ivo, "inv")


def test_quantize_nonfinite_sets_status():
    X = torch.ones(4, 100)
    X[2, 50] = float("inf")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsg.quantize_rows(X.cuda(), dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) & bsg.DSTATUS_NONFINITE
    st.zero_()
    bsg.quantize_cols(X.cuda(), dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) & bsg.DSTATUS_NONFINITE
    st.zero_()
    bsg.quantize_rows(torch.ones(4, 100, device="cuda"), dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


@pytest.mark.parametrize("case", G.row_cases(), ids=lambda c: c.name)
def test_gate_rows_on_gpu(orc, case):
    """The GPU takes the spec's answer on inputs where a variant differs."""
    row = np.tile(case.row, (3, 1))
    Q, sc, iv = bsg.quantize_rows(dev(row))
    assert [list(r) for r in host(Q).astype(int)] == [case.spec_q] * 3
    assert all(int(b) == case.spec_scale for b in u32(host(sc)))
    Qc, scc, _ = bsg.quantize_cols(dev(np.ascontiguousarray(row.T)))
    assert [list(r) for r in host(Qc).T.astype(int)] == [case.spec_q] * 3


def test_gate_epilogue_on_gpu():
    for c in G.epi_cases():
        C = bsg.epilogue(dev(np.array([[c.s]], np.int32)), dev(np.array([c.a], np.uint32).view(np.float32)),
                         dev(np.array([c.b], np.uint32).view(np.float32)))
        assert int(u32(host(C))[0, 0]) == c.spec, c.name


def test_epilogue_unit_million_triples(orc):
    from test_oracle_epilogue import epilogue_cases
    S, sa, sb = epilogue_cases(7, 1000, 1000)
    for relu in (False, True):
        C = bsg.epilogue(dev(S), dev(sa), dev(sb), relu=relu)
        Co = orc.epilogue(S, sa, sb, relu=relu)
        assert_bits_equal(host(C), Co, f"epilogue relu={relu}", nan_equal=True)
    # the grid reaches -0, subnormal and infinite outputs
    C0 = host(bsg.epilogue(dev(S), dev(sa), dev(sb), relu=False))
    b = u32(C0)
    assert (b == 0x80000000).any()
    assert ((b & 0x7F800000) == 0).any() and ((b & 0x7FFFFF) != 0).any()
    assert np.isinf(C0).any()


@pytest.mark.parametrize("shape", [(0, 5), (1, 1), (3, 7), (16, 16), (64, 64), (37, 53),
                                   (1024, 1024), (333, 1000), (2048, 3000)])
def test_hash_f32(orc, shape):
    C = np.random.default_rng(shape[0] + shape[1]).standard_normal(shape).astype(np.float32)
    if C.size:
        C.reshape(-1)[0] = -0.0
    assert bsg.hash_f32(torch.from_numpy(C).cuda()) == orc.hash_f32(C)


def test_hash_strided_rows(orc):
    big = torch.randn(50, 80, device="cuda")
    view = big[:, :61]
    lib = bsg.load()
    import ctypes
    out = torch.empty(32, dtype=torch.uint8, device="cuda")
    ws = torch.empty(lib.bsg_hash_f32_workspace_size(50, 61), dtype=torch.uint8, device="cuda")
    rc = lib.bsg_hash_f32(ctypes.c_void_p(big.data_ptr()), 50, 61, 80, ctypes.c_void_p(out.data_ptr()),
                          ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert bytes(out.cpu().tolist()) == orc.hash_f32(view.cpu().numpy())


def test_scale_derivation_selftest_exhaustive():
    """The device's f32 scale derivation equals its own f64 definition for
    every finite non-negative absmax bit pattern."""
    assert bsg.selftest_scales(0, 0x7F7FFFFF) == 0


@pytest.mark.parametrize("rows,cols,ldx", [(3, 20001, 20004), (40, 50304, 50304), (1, 16385, 16388)],
                         ids=lambda v: str(v))
def test_quantize_wide_rows_strided(orc, rows, cols, ldx):
    """Rows longer than 16384 columns (maxima by segments, then one streaming
    pass), with a row stride past the row and a tail that is not a whole
    float4: codes, scales and inv against the oracle, and the padding of X
    never read into the result."""
    import ctypes
    Xfull = inputs.adversarial(rows, ldx, rows + cols).numpy()
    Xfull[:, cols:] = np.float32(1e30)          # padding that must not count
    X = np.ascontiguousarray(Xfull[:, :cols])
    Xd = dev(Xfull)
    Q = torch.zeros(rows, cols, dtype=torch.int8, device="cuda")
    sc = torch.zeros(rows, dtype=torch.float32, device="cuda")
    iv = torch.zeros(rows, dtype=torch.float32, device="cuda")
    rc = bsg.load().bsg_quantize_rows(ctypes.c_void_p(Xd.data_ptr()), rows, cols, ldx,
                                      ctypes.c_void_p(Q.data_ptr()), cols,
                                      ctypes.c_void_p(sc.data_ptr()), ctypes.c_void_p(iv.data_ptr()),
                                      None, None)
    assert rc == 0
    torch.cuda.synchronize()
    Qo, sco, ivo, _ = orc.quantize_rows(X)
    assert_bits_equal(host(Q), Qo, "Q")
    assert_bits_equal(host(sc), sco, "scale")
    assert_bits_equal(host(iv), ivo, "inv")
