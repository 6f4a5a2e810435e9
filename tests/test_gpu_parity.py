"""GPU parity of the whole unit (bsgemm_i8 and friends) against the CPU
oracle, bitwise, through the C ABI.

Rule: "Verification -- why you can trust the numbers", section "The verified
INT8 units" (steps 1-3) and section "Layer 1: exact init gates": kernel and
mirror are compared on a sweep of shapes, ragged ones included, int32
accumulators exactly and f32 outputs at the bit level.

Sizes: small shapes are compared in full; the full-size workloads are run in
the same launch configuration the benchmark times and compared in full
where the oracle takes seconds, else on sampled cells the oracle computes one
by one (``orc.bsgemm_cells``) plus properties that hold at any size.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal, dev, host, u32
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu


def gpu_unit(A, B, relu=False, transA=False, transB=False):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if transA or transB:
        C = bsg.bsgemm_i8_ex(dev(A), dev(B), transA=transA, transB=transB, relu=relu, dstatus=st)
    else:
        C = bsg.bsgemm_i8(dev(A), dev(B), relu=relu, dstatus=st)
    torch.cuda.synchronize()
    return host(C), int(st.item())


def sample_cells(M, N, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.concatenate([rng.integers(0, M, n), [0, M - 1, M - 1, 0]])
    cols = np.concatenate([rng.integers(0, N, n), [0, N - 1, 0, N - 1]])
    return rows, cols


# ---------------------------------------------------------------- small, full
def test_square_256(orc):
    A = inputs.normal((256, 256), 1.0, 0).numpy()
    B = inputs.normal((256, 256), 1.0, 100).numpy()
    C, st = gpu_unit(A, B)
    assert st == 0
    Co, so = orc.bsgemm_i8(A, B)
    assert_bits_equal(C, Co, "256^3")


@pytest.mark.parametrize("idx", range(64))
def test_tiny_shapes(orc, idx):
    M, N, K, seed = inputs.tiny_shapes()[idx]
    A = inputs.normal((M, K), 1.0, seed).numpy()
    B = inputs.normal((K, N), 1.0, seed + 50_000).numpy()
    relu = bool(idx % 2)
    C, st = gpu_unit(A, B, relu)
    assert st == 0
    Co, _ = orc.bsgemm_i8(A, B, relu)
    assert_bits_equal(C, Co, f"tiny {M}x{N}x{K}")


@pytest.mark.parametrize("shape", [(128, 256, 64), (129, 257, 65), (1, 300, 5), (300, 1, 7),
                                   (255, 511, 1023), (200, 300, 1024), (130, 260, 1025),
                                   (77, 513, 1040), (96, 96, 2049), (250, 260, 3000),
                                   (64, 64, 4097), (1000, 40, 8)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("relu", [False, True])
def test_ragged_shapes_full(orc, shape, relu):
    M, N, K = shape
    A = inputs.uniform((M, K), -1, 1, M + K).numpy()
    B = inputs.uniform((K, N), -1, 1, N + 3 * K).numpy()
    C, st = gpu_unit(A, B, relu)
    assert st == 0
    Co, _ = orc.bsgemm_i8(A, B, relu)
    assert_bits_equal(C, Co, f"{shape} relu={relu}")


@pytest.mark.parametrize("shape", [(128, 256, 64), (33, 70, 17), (256, 512, 1024),
                                   (130, 300, 1040), (129, 257, 2500), (64, 256, 5000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_s32_accumulators(orc, shape):
    M, N, K = shape
    rng = np.random.default_rng(M * N + K)
    Aq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    Bq = rng.integers(-127, 128, (K, N)).astype(np.int8)
    S = host(bsg.gemm_s32(dev(Aq), dev(Bq)))
    So, st = orc.gemm_s32(Aq, Bq)
    assert_bits_equal(S, So, "S")


@pytest.mark.parametrize("K", [1, 16, 1023, 1024, 1025, 1040, 1041, 2048, 4096, 8192, 16384,
                               133144])
def test_exactness_saturated_and_cancelling(orc, K):
    """The fp32 tensor-core chunks must stay exact: saturated +-127 operands
    (the largest partial sums), alternating-sign cancellation, and runs that
    build up to the 2^24 edge and come back."""
    M, N = 128, 256
    Aq = np.full((M, K), 127, np.int8)
    Bq = np.full((K, N), 127, np.int8)
    Aq[1::4] = -127
    Bq[:, 1::3] = -127
    alt = np.where(np.arange(K) % 2 == 0, 127, -127).astype(np.int8)
    Aq[2::4] = alt
    Bq[:, 2::3] = alt[:, None]
    # a run that climbs for the first half of K and falls for the second
    Aq[3] = np.where(np.arange(K) < K // 2, 127, -127)
    S = host(bsg.gemm_s32(dev(Aq), dev(Bq)))
    So, st = orc.gemm_s32(Aq, Bq)
    assert st == 0
    assert_bits_equal(S, So, f"K={K}")
    assert int(So[0, 0]) == 127 * 127 * K


@pytest.mark.parametrize("M", [5, 129])
def test_unit_at_max_k(orc, M):
    """The whole f32 unit at K = BSG_MAX_K: A's rows beyond 16384 columns
    (segmented maxima, then the streaming pass), B's 133144-row columns (the
    one-read column quantize), and saturated rows whose integer sums reach
    127^2 K, just inside int32; C bitwise the oracle's."""
    K, N = bsg.MAX_K, 9
    rng = np.random.default_rng(K + M)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    A[0] = 1.0                                  # codes 127 everywhere
    A[1] = np.where(np.arange(K) % 2 == 0, 1.0, -1.0)
    B[:, 0] = 1.0
    B[:, 1] = np.where(np.arange(K) % 2 == 0, 1.0, -1.0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = bsg.bsgemm_i8(dev(A), dev(B), dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Co, rc = orc.bsgemm_i8(A, B, False)
    assert rc == 0
    assert_bits_equal(host(C), Co, f"M={M} K={K}")
    # S[0][0] = 127^2 K exactly; C = S * (1/127) * (1/127) in f32 steps
    assert Co[0, 0] == np.float32(np.float32(np.float32(127 * 127 * K) * np.float32(1 / 127))
                                  * np.float32(1 / 127))


def test_max_k_limit_and_status():
    A = torch.ones(2, 8, device="cuda")
    B = torch.ones(8, 2, device="cuda")
    lib = bsg.load()
    import ctypes
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    rc = lib.bsgemm_i8(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()), 2, 2,
                       bsg.MAX_K + 1, 0, ctypes.c_void_p(A.data_ptr()),
                       ctypes.c_void_p(ws.data_ptr()), ws.numel(), None, None)
    assert rc == 2   # BSG_ERR_K_TOO_LARGE
    rc = lib.bsgemm_i8(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()), 2, 2, 8, 0,
                       ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(ws.data_ptr()), 16, None, None)
    assert rc == 3   # workspace too small


def test_nonfinite_input_sets_status():
    A = inputs.normal((64, 64), 1.0, 1).numpy()
    A[5, 5] = np.nan
    _, st = gpu_unit(A, inputs.normal((64, 32), 1.0, 2).numpy())
    assert st & bsg.DSTATUS_NONFINITE


# ----------------------------------------------------- adversarial values
def test_adversarial_block_1024(orc):
    A = inputs.adversarial(1024, 1024, 10).numpy()
    B = inputs.adversarial(1024, 1024, 11, along_rows=False).numpy()
    for relu in (False, True):
        C, st = gpu_unit(A, B, relu)
        assert st == 0
        Co, _ = orc.bsgemm_i8(A, B, relu)
        assert_bits_equal(C, Co, f"adversarial relu={relu}")


def test_adversarial_reaches_edge_cases(orc):
    A = inputs.adversarial(300, 200, 12).numpy()
    B = inputs.adversarial(150, 200, 13, along_rows=False).numpy()
    C, st = gpu_unit(A, B)
    Co, _ = orc.bsgemm_i8(A, B)
    assert_bits_equal(C, Co, "adversarial 300x150x200")
    assert np.isinf(C).any() and (u32(C) == 0).any()


# ------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["qkv", "fc", "proj"])
def test_gpt2_linears_full(orc, name):
    A, B, relu = inputs.gpt2_linear_inputs(name)
    A, B = A.numpy(), B.numpy()
    C, st = gpu_unit(A, B, relu)
    assert st == 0
    Co, so = orc.bsgemm_i8(A, B, relu)
    assert_bits_equal(C, Co, name)


def test_lm_head_full(orc):
    _, M, N, K, relu, seed = inputs.LM_HEAD
    A = inputs.gpt2_activations(M, K, seed, outlier_frac=0.0).numpy()
    B = inputs.gpt2_weights(K, N, seed).numpy()
    C, st = gpu_unit(A, B, relu)
    assert st == 0
    Co, _ = orc.bsgemm_i8(A, B, relu)
    assert_bits_equal(C, Co, "lm_head")
    assert np.isfinite(C).all()


@pytest.mark.parametrize("which", [0, 1, 2], ids=["fwd", "dgrad", "wgrad"])
def test_train_trio_full(orc, which):
    X, W, dY = (t.numpy() for t in inputs.train_trio())
    name, M, N, K, tA, tB = inputs.TRAIN_TRIO[which]
    if name == "fwd":
        A, B = X, W
    elif name == "dgrad":
        A, B = dY, W            # B stored N x K (W is 768 x 3072 = N x K): op(B) = W^T
    else:
        A, B = X, dY            # A stored K x M: op(A) = X^T
    C, st = gpu_unit(A, B, transA=tA, transB=tB)
    assert st == 0
    Am = np.ascontiguousarray(A.T) if tA else A
    Bm = np.ascontiguousarray(B.T) if tB else B
    assert Am.shape == (M, K) and Bm.shape == (K, N)
    Co, so = orc.bsgemm_i8(Am, Bm)
    assert_bits_equal(C, Co, name)


@pytest.mark.parametrize("name", [g[0] for g in inputs.LARGE_GEMMS])
def test_large_gemms_full(orc, name):
    """The benchmark's GEMMs -- 4096^3, 8192^3, 16384^3 of U(-1, 1) values and
    the ragged 4097 x 12289 x 8191 with the adversarial mixes -- compared with
    the oracle over the whole of C, bit for bit."""
    A, B, relu = inputs.large_gemm_inputs(name)
    A, B = A.numpy(), B.numpy()
    C, st = gpu_unit(A, B, relu)
    assert st == 0
    Co, _ = orc.bsgemm_i8(A, B, relu)
    assert_bits_equal(C, Co, name)
    if name == "ragged_adversarial":
        # the mix reaches what it is meant to: overflow to +-Inf from the 1e30
        # vectors, exact zeros from the zero and 1e-30 ones
        assert np.isposinf(C).any() and np.isneginf(C).any()
        assert (u32(C) == 0).any()


@pytest.mark.parametrize("name", ["sq4096", "sq8192", "ragged_adversarial"])
def test_large_int32_accumulators_full(orc, name):
    """The contraction alone at the benchmark's sizes: the oracle's int8
    codes of A and B through bsg_gemm_s32 (the same tensor-core kernel,
    int32 S stored instead of the epilogue), compared with the oracle's
    exact S over the whole matrix."""
    A, B, _ = inputs.large_gemm_inputs(name)
    Aq, _, _, _ = orc.quantize_rows(A.numpy())
    Bq, _, _, _ = orc.quantize_cols(B.numpy())
    S = host(bsg.gemm_s32(dev(Aq), dev(Bq)))
    So, _ = orc.gemm_s32(Aq, Bq)
    assert_bits_equal(S, So, name + " S")


@pytest.mark.parametrize("shape", [(384, 512, 6400), (8192, 768, 3072), (1024, 1024, 1024),
                                   (1280, 2560, 1100), (640, 300, 4097), (150 * 128, 256, 768)],
                         ids=lambda s: "x".join(map(str, s)))
def test_split_tiles_exact_and_deterministic(orc, shape):
    """Shapes whose tiles are split along K across CTAs (and across exact
    chunks): the int32 sums combined from several CTAs equal the oracle's,
    and two runs give the same bits."""
    M, N, K = shape
    rng = np.random.default_rng(M + N + K)
    Aq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    Bq = rng.integers(-127, 128, (K, N)).astype(np.int8)
    Aq[0] = 127
    Bq[:, 0] = 127
    S1 = host(bsg.gemm_s32(dev(Aq), dev(Bq)))
    S2 = host(bsg.gemm_s32(dev(Aq), dev(Bq)))
    np.testing.assert_array_equal(S1, S2)
    if M * N * K <= 4_000_000_000:
        So, st = orc.gemm_s32(Aq, Bq)
        assert_bits_equal(S1, So, f"S {shape}")
    else:
        rows, cols = sample_cells(M, N, 2000, 3)
        exact = np.einsum("ik,ki->i", Aq[rows].astype(np.int64), Bq[:, cols].astype(np.int64))
        np.testing.assert_array_equal(S1[rows, cols].astype(np.int64), exact)
