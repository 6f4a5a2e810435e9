"""Layer-5 properties on the GPU path, through the C ABI.

"Verification -- why you can trust the numbers", section "Layer 5":
relations (row permutation permutes outputs; a zero row yields zeros;
batches decompose; single-cell sensitivity) and two absolutes (fused ReLU
never negative; at unit scales the output is the exact integer dot
product).  These hold at any size, so they also cover shapes too large for a
full oracle comparison.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal, dev, host, u32
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu


def run(A, B, relu=False):
    return host(bsg.bsgemm_i8(dev(A), dev(B), relu=relu))


@pytest.fixture(scope="module")
def case():
    A = inputs.gpt2_activations(1024, 768, 21).numpy()
    B = inputs.gpt2_weights(768, 640, 21).numpy()
    return A, B, run(A, B)


def test_row_and_column_permutation(case):
    A, B, C = case
    rng = np.random.default_rng(0)
    pr, pc = rng.permutation(A.shape[0]), rng.permutation(B.shape[1])
    assert_bits_equal(run(A[pr], B[:, pc]), C[pr][:, pc], "permuted")


def test_zero_rows_and_columns(case):
    A, B, _ = case
    A2, B2 = A.copy(), B.copy()
    A2[[3, 500, 1023]] = 0.0
    A2[7] = -0.0
    B2[:, [0, 255, 639]] = 0.0
    for relu in (False, True):
        C = run(A2, B2, relu)
        for r in (3, 500, 1023, 7):
            assert not u32(C[r]).any()
        for c in (0, 255, 639):
            assert not u32(C[:, c]).any()


def test_batches_decompose(case):
    A, B, C = case
    parts = [run(A[a:b], B) for a, b in ((0, 1), (1, 129), (129, 700), (700, 1024))]
    assert_bits_equal(np.concatenate(parts), C, "row batches")
    cparts = [run(A, B[:, a:b]) for a, b in ((0, 256), (256, 257), (257, 640))]
    assert_bits_equal(np.concatenate(cparts, axis=1), C, "column batches")


def test_single_cell_sensitivity(case):
    A, B, C = case
    A2 = A.copy()
    A2[300, 10] += 2.5
    d = u32(run(A2, B)) != u32(C)
    assert d[300].any() and not np.delete(d, 300, axis=0).any()
    B2 = B.copy()
    B2[100, 77] -= 0.5
    d = u32(run(A, B2)) != u32(C)
    assert d[:, 77].any() and not np.delete(d, 77, axis=1).any()


def test_relu_never_negative():
    A = inputs.adversarial(700, 900, 31).numpy()
    B = inputs.adversarial(500, 900, 32, along_rows=False).numpy()
    C = run(A, B, relu=True)
    assert not (u32(C) >> 31).any()
    C0 = run(A, B, relu=False)
    assert (C0 < 0).any()


@pytest.mark.parametrize("K", [700, 1024, 3000])
def test_unit_scales_exact_integer_dot(K):
    rng = np.random.default_rng(K)
    M, N = 300, 260
    A = rng.integers(-127, 128, (M, K)).astype(np.float32)
    B = rng.integers(-127, 128, (K, N)).astype(np.float32)
    A[:, 0] = 127
    B[0, :] = -127
    exact = A.astype(np.int64) @ B.astype(np.int64)
    C = run(A, B)
    # exact while |dot| < 2^24; beyond, f32(S) is the correctly rounded dot
    np.testing.assert_array_equal(C, exact.astype(np.float32))
    S = host(bsg.gemm_s32(dev(A.astype(np.int8)), dev(B.astype(np.int8))))
    np.testing.assert_array_equal(S.astype(np.int64), exact)


def test_probe_hash_is_deterministic_and_seeded():
    h0 = bsg.probe_hash(0)
    assert bsg.probe_hash(0) == h0
    assert bsg.probe_hash(1) != h0


def test_probe_hash_golden():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "probe_hash.txt")
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            seed, M, N, K, h = line.split()
            assert bsg.probe_hash(int(seed), int(M), int(N), int(K)).hex() == h, line


def test_host_buffer_entry_point(orc):
    A = inputs.gpt2_activations(512, 768, 41).numpy()
    B = inputs.gpt2_weights(768, 300, 41).numpy()
    Ah = torch.from_numpy(A).pin_memory()
    Bh = torch.from_numpy(B).pin_memory()
    C, st = bsg.bsgemm_i8_host(Ah, Bh, relu=True)
    assert st == 0
    Co, _ = orc.bsgemm_i8(A, B, True)
    assert_bits_equal(C.numpy(), Co, "host entry point")


@pytest.mark.parametrize("M,N,K", [(3000, 257, 1100), (8192, 2304, 768), (100, 33, 65),
                                   (2049, 64, 3072)])
def test_host_buffer_entry_point_chunked(orc, M, N, K):
    """The host entry point moves A in row chunks and overlaps copies with the
    kernels: ragged chunk counts and a last partial chunk give the same bits."""
    A = inputs.gpt2_activations(M, K, M + K).numpy()
    B = inputs.gpt2_weights(K, N, N).numpy()
    Ah = torch.from_numpy(A).pin_memory()
    Bh = torch.from_numpy(B).pin_memory()
    C, st = bsg.bsgemm_i8_host(Ah, Bh, relu=False)
    assert st == 0
    if M * N * K <= 3000 * 257 * 1100:
        Co, _ = orc.bsgemm_i8(A, B, False)
        assert_bits_equal(C.numpy(), Co, f"host {M}x{N}x{K}")
    else:
        Cd = bsg.bsgemm_i8(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
        torch.cuda.synchronize()
        assert_bits_equal(C.numpy(), Cd.cpu().numpy(), "host vs device entry point")


def test_host_batch_matches_the_oracle(orc):
    """Several units in one pipelined host call: each C is the oracle's, the
    items sharing one B and differing in shape, chunk count and ReLU."""
    shapes = [(700, 130, 1100, True), (2600, 257, 768, False), (64, 33, 65, True),
              (1300, 130, 1100, False)]
    data = []
    for i, (M, N, K, relu) in enumerate(shapes):
        A = inputs.gpt2_activations(M, K, 60 + i).numpy()
        B = inputs.gpt2_weights(K, N, 70 + i).numpy()
        data.append((A, B, relu))
    # items 0 and 3 share B (read-only inputs may be shared)
    data[3] = (data[3][0], data[0][1], data[3][2])
    items = [(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(), relu)
             for A, B, relu in data]
    outs, st = bsg.bsgemm_i8_host_batch(items)
    assert st == 0
    for i, ((A, B, relu), C) in enumerate(zip(data, outs)):
        Co, _ = orc.bsgemm_i8(A, B, relu)
        assert_bits_equal(C.numpy(), Co, f"batch item {i}")


def test_host_batch_gpt2_linears_equal_device_entry_point():
    """The three GPT-2-small linears at M = 8192 in one batch, as the
    end-to-end measurement runs them: bit for bit the device entry point."""
    items, dev_out = [], []
    for name, M, N, K, relu, seed in inputs.GPT2_LINEARS:
        A, B, _ = inputs.gpt2_linear_inputs(name)
        items.append((A.pin_memory(), B.pin_memory(), relu))
        dev_out.append(bsg.bsgemm_i8(A.cuda(), B.cuda(), relu=relu))
    outs, st = bsg.bsgemm_i8_host_batch(items)
    torch.cuda.synchronize()
    assert st == 0
    for (name, *_), C, Cd in zip(inputs.GPT2_LINEARS, outs, dev_out):
        assert_bits_equal(C.numpy(), Cd.cpu().numpy(), f"batch {name}")


def test_host_batch_reports_nonfinite_input():
    A0 = inputs.normal((300, 200), 1.0, 1)
    A1 = inputs.normal((300, 200), 1.0, 2)
    A1[7, 9] = float("inf")
    B = inputs.normal((200, 100), 1.0, 3)
    items = [(A0.pin_memory(), B.pin_memory(), False), (A1.pin_memory(), B.pin_memory(), False)]
    outs, st = bsg.bsgemm_i8_host_batch(items)
    assert st == bsg.DSTATUS_NONFINITE


def test_host_batch_order_does_not_change_results():
    """The batch call reorders its items for the host link; each C still
    belongs to its own item, bit for bit."""
    data = []
    for i, (M, N, K) in enumerate([(2100, 64, 3000), (700, 900, 256), (1500, 1200, 300)]):
        A = inputs.gpt2_activations(M, K, 90 + i)
        B = inputs.gpt2_weights(K, N, 95 + i)
        data.append((A.pin_memory(), B.pin_memory(), i == 1))
    fwd, _ = bsg.bsgemm_i8_host_batch(data)
    rev, _ = bsg.bsgemm_i8_host_batch(list(reversed(data)))
    for i, C in enumerate(fwd):
        Cd = bsg.bsgemm_i8(data[i][0].cuda(), data[i][1].cuda(), relu=data[i][2])
        torch.cuda.synchronize()
        assert_bits_equal(C.numpy(), Cd.cpu().numpy(), f"item {i}")
        assert_bits_equal(rev[len(data) - 1 - i].numpy(), C.numpy(), f"reversed item {i}")
