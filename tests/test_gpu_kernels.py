"""Every GEMM kernel instantiation against the oracle, bitwise.

The library picks one of eight tensor-core kernels per problem: a 128-row
tile on one SM or a 256-row tile on a pair of SMs (M > 128), each at tile
width 64, 128, 192 or 256.  The workloads exercise only the choices the
schedule makes for them, so these tests force each kernel in turn (the
BSG_GEMM_PAIR and BSG_GEMM_BN environment switches, read on every call) on
ragged shapes -- partial m-blocks, a pair whose second CTA has no rows,
partial n-tiles including N in (192, 256], one and several exact 1024-deep
K chunks -- and compare C (and the int32 accumulators) with the oracle.

Rule: "Verification -- why you can trust the numbers", section "The verified
INT8 units": the result is defined independently of tiling, so every
schedule must reproduce the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal, dev, host
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu

SHAPES = [(300, 200, 100), (129, 257, 1025), (520, 383, 2100), (256, 256, 64), (640, 250, 960),
          (100, 700, 1030)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("bn", [64, 128, 192, 256])
@pytest.mark.parametrize("pair", [True, False], ids=["pair", "single"])
def test_forced_kernel_matches_oracle(orc, monkeypatch, shape, bn, pair):
    monkeypatch.setenv("BSG_GEMM_BN", str(bn))
    monkeypatch.setenv("BSG_GEMM_PAIR", "1" if pair else "0")
    M, N, K = shape
    relu = (M + bn) % 2 == 1
    A = inputs.normal((M, K), 1.0, M * 31 + K).numpy()
    B = inputs.normal((K, N), 1.0, N * 17 + K).numpy()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = bsg.bsgemm_i8(dev(A), dev(B), relu=relu, dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Co, _ = orc.bsgemm_i8(A, B, relu)
    assert_bits_equal(host(C), Co, f"{shape} bn={bn} pair={pair} relu={relu}")


@pytest.mark.parametrize("bn", [64, 128, 192, 256])
@pytest.mark.parametrize("pair", [True, False], ids=["pair", "single"])
def test_forced_kernel_int32_accumulators(orc, monkeypatch, bn, pair):
    monkeypatch.setenv("BSG_GEMM_BN", str(bn))
    monkeypatch.setenv("BSG_GEMM_PAIR", "1" if pair else "0")
    M, N, K = 390, 230, 2200
    rng = np.random.default_rng(bn + 7 * pair)
    Aq = rng.integers(-127, 128, (M, K), dtype=np.int64).astype(np.int8)
    Bq = rng.integers(-127, 128, (K, N), dtype=np.int64).astype(np.int8)
    S = bsg.gemm_s32(dev(Aq), dev(Bq))
    torch.cuda.synchronize()
    want, _ = orc.gemm_s32(Aq, Bq)
    assert_bits_equal(host(S), want, f"S bn={bn} pair={pair}")


def test_switches_are_read_per_call(orc, monkeypatch):
    """The same inputs through two different kernels give the same bits."""
    M, N, K = 512, 384, 1500
    A = inputs.uniform((M, K), -1, 1, 5).numpy()
    B = inputs.uniform((K, N), -1, 1, 6).numpy()
    outs = []
    for bn, pair in ((256, "1"), (64, "0")):
        monkeypatch.setenv("BSG_GEMM_BN", str(bn))
        monkeypatch.setenv("BSG_GEMM_PAIR", pair)
        outs.append(host(bsg.bsgemm_i8(dev(A), dev(B))))
    torch.cuda.synchronize()
    assert_bits_equal(outs[0], outs[1], "256/pair vs 64/single")


@pytest.mark.parametrize("M,N,K", [(64, 300, 4097), (130, 129, 5000), (40, 257, 8191),
                                   (33, 1000, 9000)], ids=lambda v: str(v))
def test_long_columns_two_pass_operand(orc, M, N, K):
    """Columns longer than the strip kernel's 4096 rows go through the
    two-pass column quantize into the f16 operand (a transposing tile);
    B's columns carry the adversarial kinds, K is odd or ragged."""
    A = inputs.normal((M, K), 1.0, M + K).numpy()
    B = inputs.adversarial(N, K, N + K, along_rows=False).numpy()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = bsg.bsgemm_i8(dev(A), dev(B), dstatus=st)
    torch.cuda.synchronize()
    Co, _ = orc.bsgemm_i8(A, B, False)
    assert_bits_equal(host(C), Co, f"{M}x{N}x{K}")


def test_long_columns_transposed_a(orc):
    """op(A) = A^T of a stored K x M matrix with K > 4096: A's per-row
    quantize of op(A) is a column quantize of the stored matrix."""
    M, N, K = 200, 96, 6000
    At = inputs.gpt2_activations(K, M, 17).numpy()     # stored K x M
    B = inputs.gpt2_weights(K, N, 18).numpy()
    C = bsg.bsgemm_i8_ex(dev(At), dev(B), transA=True)
    torch.cuda.synchronize()
    Co, _ = orc.bsgemm_i8(np.ascontiguousarray(At.T), B, False)
    assert_bits_equal(host(C), Co, "transA K=6000")


COL_SHAPES = [(64, 300, 4097), (130, 129, 5000), (40, 257, 8191), (33, 1000, 9000),
              (24, 96, 16384), (50, 77, 1000), (3, 5, 7)]


@pytest.mark.parametrize("path", ["strip", "lag", "twopass", ""])
@pytest.mark.parametrize("M,N,K", COL_SHAPES, ids=lambda v: str(v))
def test_every_column_quantize_path_operand(orc, monkeypatch, path, M, N, K):
    """Each column-quantize path (register strips in clusters, the one-read
    list of max and quantize items, two passes) forced in turn into the
    GEMM's f16 operand, on columns with the adversarial kinds, short, long,
    odd and ragged: C bitwise equal to the oracle's.  Strips do not apply
    beyond 4096 rows; those shapes take the one-read path unless two passes
    are forced."""
    monkeypatch.setenv("BSG_COLS_PATH", path)
    A = inputs.normal((M, K), 1.0, M + K).numpy()
    B = inputs.adversarial(N, K, N + K + 1, along_rows=False).numpy()
    C = bsg.bsgemm_i8(dev(A), dev(B))
    torch.cuda.synchronize()
    Co, _ = orc.bsgemm_i8(A, B, False)
    assert_bits_equal(host(C), Co, f"{path} {M}x{N}x{K}")


@pytest.mark.parametrize("lag", ["1", "2", "7", "4096"])
@pytest.mark.parametrize("M,N,K", [(64, 999, 5000), (40, 129, 16384), (8, 3001, 600)],
                         ids=lambda v: str(v))
def test_one_read_column_quantize_any_lag(orc, monkeypatch, lag, M, N, K):
    """The one-read column quantize with its lag forced from one panel (each
    panel's quantize items right after the next panel's max items) to more
    panels than there are (all max items first): the same bits every time,
    the oracle's.  N is odd, so B's rows are not 16-byte aligned, which the
    path's scalar loads take as they are."""
    monkeypatch.setenv("BSG_COLS_PATH", "lag")
    monkeypatch.setenv("BSG_COLQ_LAG", lag)
    A = inputs.normal((M, K), 1.0, 3 * M + K).numpy()
    B = inputs.adversarial(N, K, N + K + 5, along_rows=False).numpy()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = bsg.bsgemm_i8(dev(A), dev(B), dstatus=st)
    torch.cuda.synchronize()
    Co, _ = orc.bsgemm_i8(A, B, False)
    assert_bits_equal(host(C), Co, f"lag {lag} {M}x{N}x{K}")
    assert not int(st.item()) & 2, "a bounded wait expired"


@pytest.mark.parametrize("path", ["twopass", ""])
@pytest.mark.parametrize("R,Ncol", [(5000, 129), (4100, 33), (3000, 40), (300, 17), (7, 3)],
                         ids=lambda v: str(v))
def test_every_column_quantize_path_int8(orc, monkeypatch, path, R, Ncol):
    """The int8 column quantize (codes in X's layout, scales and inv) on
    every path (clusters up to 3072 rows unless two passes are forced),
    against the oracle, bitwise."""
    monkeypatch.setenv("BSG_COLS_PATH", path)
    X = inputs.adversarial(Ncol, R, R + Ncol, along_rows=False).numpy()
    Q, sc, iv = bsg.quantize_cols(dev(X))
    Qo, sco, ivo, _ = orc.quantize_cols(X)
    assert_bits_equal(host(Q), Qo, "Q")
    assert_bits_equal(host(sc), sco, "scale")
    assert_bits_equal(host(iv), ivo, "inv")


@pytest.mark.parametrize("group,snake", [(1, "1"), (3, "1"), (8, "1"), (8, "0"), (64, "1")])
def test_tile_raster_does_not_change_results(orc, monkeypatch, group, snake):
    """The order in which tiles are handed out (BSG_GEMM_GROUP m-units per
    raster group, serpentine or not) changes which CTA computes which tile
    and when, never a bit of C."""
    monkeypatch.setenv("BSG_GEMM_GROUP", str(group))
    monkeypatch.setenv("BSG_GEMM_SNAKE", snake)
    M, N, K = 1300, 1100, 2100
    A = inputs.normal((M, K), 1.0, 31).numpy()
    B = inputs.normal((K, N), 0.1, 32).numpy()
    C = bsg.bsgemm_i8(dev(A), dev(B), relu=True)
    torch.cuda.synchronize()
    Co, _ = orc.bsgemm_i8(A, B, True)
    assert_bits_equal(host(C), Co, f"group {group}")


UNALIGNED_PATHS = {"shift": {}, "peel": {"BSG_ROWS_SHIFT": "0"},
                   "scalar": {"BSG_ROWS_SHIFT": "0", "BSG_ROWS_PEEL": "0"}}


@pytest.mark.parametrize("path", list(UNALIGNED_PATHS))
@pytest.mark.parametrize("rows,cols", [(33, 65), (300, 1001), (17, 8191), (5, 20001), (64, 70),
                                       (40, 2049), (9, 12287), (6, 16383), (3, 8193)],
                         ids=lambda v: str(v))
def test_unaligned_rows_every_path(orc, monkeypatch, path, rows, cols):
    """Rows that are not 16-byte aligned (ldx % 4 != 0): the register-resident
    kernel that loads each row from its first 16-byte boundary (long rows),
    the kernel that peels each row to that boundary and the scalar one,
    forced in turn, for the int8 API and inside the unit (the f16 operand),
    against the oracle."""
    for k, v in UNALIGNED_PATHS[path].items():
        monkeypatch.setenv(k, v)
    X = inputs.adversarial(rows, cols, rows * 7 + cols).numpy()
    Q, sc, iv = bsg.quantize_rows(dev(X))
    Qo, sco, ivo, _ = orc.quantize_rows(X)
    assert_bits_equal(host(Q), Qo, "Q")
    assert_bits_equal(host(sc), sco, "scale")
    assert_bits_equal(host(iv), ivo, "inv")
    B = inputs.normal((cols, 40), 0.1, cols).numpy()
    C = bsg.bsgemm_i8(dev(X), dev(B))
    torch.cuda.synchronize()
    Co, _ = orc.bsgemm_i8(X, B, False)
    assert_bits_equal(host(C), Co, "C")


@pytest.mark.parametrize("pad", [1, 2, 3])
@pytest.mark.parametrize("cols", [2049, 6000, 8192, 12001, 16384])
def test_unaligned_rows_int8_aligned_output(orc, pad, cols):
    """The int8 API with X's rows not 16-byte aligned (ldx = cols + pad) and
    Q's rows 16-byte aligned (ldq a multiple of 16), the layout the
    register-resident kernel takes for the int8 codes: codes, scales and inv
    bitwise the oracle's, and Q's padding columns untouched."""
    import ctypes
    rows = 21
    ldx, ldq = cols + pad, (cols + 15) // 16 * 16 + 16
    Xw = inputs.adversarial(rows, ldx, cols + pad).numpy()
    X = np.ascontiguousarray(Xw[:, :cols])
    dX = dev(Xw)
    Q = torch.full((rows, ldq), 0x5A, dtype=torch.int8, device="cuda")
    sc = torch.empty(rows, dtype=torch.float32, device="cuda")
    iv = torch.empty(rows, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = bsg.load()
    rc = lib.bsg_quantize_rows(ctypes.c_void_p(dX.data_ptr()), rows, cols, ldx,
                               ctypes.c_void_p(Q.data_ptr()), ldq, ctypes.c_void_p(sc.data_ptr()),
                               ctypes.c_void_p(iv.data_ptr()), ctypes.c_void_p(st.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    Qo, sco, ivo, _ = orc.quantize_rows(X)
    Qh = host(Q)
    assert_bits_equal(Qh[:, :cols], Qo, "Q")
    assert (Qh[:, cols:] == 0x5A).all(), "Q's padding was written"
    assert_bits_equal(host(sc), sco, "scale")
    assert_bits_equal(host(iv), ivo, "inv")


@pytest.mark.parametrize("case", ["B long columns", "B long columns, two passes",
                                  "A unaligned long rows", "A wide rows", "A rows beyond 16384"])
def test_nonfinite_on_every_long_path_sets_status(monkeypatch, case):
    """An Inf or NaN on each long-vector quantize path (the one-read column
    list, the two passes, the register-resident unaligned rows, the wide
    rows, the segmented rows beyond 16384 columns) sets the non-finite bit,
    and no bounded wait expires."""
    M, N, K = 6, 300, 5000
    if case == "A unaligned long rows":
        K = 8191
    elif case == "A wide rows":
        K = 16384
    elif case == "A rows beyond 16384":
        K = 20000
    if case.endswith("two passes"):
        monkeypatch.setenv("BSG_COLS_PATH", "twopass")
    A = inputs.normal((M, K), 1.0, K).numpy()
    B = inputs.normal((K, N), 0.1, K + 1).numpy()
    if case.startswith("B"):
        B[4000, 17] = np.inf
    else:
        A[3, K - 9] = np.nan
        A[1, 9] = -np.inf
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsg.bsgemm_i8(dev(A), dev(B), dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) & bsg.DSTATUS_NONFINITE
    assert not int(st.item()) & 2
