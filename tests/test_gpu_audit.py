"""The live audit (bsg_audit) and the init gate (bsg_selftest) on the GPU.

Rule: "Verification -- why you can trust the numbers", section "Layer 2: the
live audit" (sampled cells of a live GEMM recomputed independently and
compared bit for bit) and section "Layer 1: exact init gates" (the kernels
checked on fixed inputs before they are trusted).

The audit must find nothing on correct outputs and must find a wrong bit.
It must also sample the cells its published rule names: SplitMix64 output
2s gives the row (mod M) and output 2s + 1 the column (mod N). That rule is
checked against the oracle's own SplitMix64.
"""
import numpy as np
import pytest
import torch

from gpu_util import dev
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu


def unit(A, B, relu=False):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = bsg.bsgemm_i8(A, B, relu=relu, dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return C


@pytest.mark.parametrize("shape,relu", [((300, 200, 100), True), ((129, 257, 1025), False),
                                        ((8192, 2304, 768), False), ((5, 7, 3), True)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_audit_finds_nothing_on_correct_output(shape, relu):
    M, N, K = shape
    A = dev(inputs.normal((M, K), 1.0, M + 1).numpy())
    B = dev(inputs.normal((K, N), 1.0, N + 2).numpy())
    C = unit(A, B, relu)
    mis = bsg.audit(A, B, C, relu=relu, seed=11, nsamples=2048)
    torch.cuda.synchronize()
    assert int(mis.item()) == 0


def test_audit_cells_follow_the_published_rule(orc):
    M, N, K = 1000, 777, 64
    A = dev(inputs.normal((M, K), 1.0, 3).numpy())
    B = dev(inputs.normal((K, N), 1.0, 4).numpy())
    C = unit(A, B)
    n = 300
    cells = torch.empty(2 * n, dtype=torch.int64, device="cuda")
    bsg.audit(A, B, C, seed=12345, nsamples=n, cells=cells)
    got = cells.cpu().numpy().reshape(n, 2)
    want = np.array([[orc.splitmix64(12345, 2 * s) % M, orc.splitmix64(12345, 2 * s + 1) % N]
                     for s in range(n)])
    assert (got == want).all()


def test_audit_finds_a_flipped_bit():
    M, N, K = 256, 256, 300
    A = dev(inputs.uniform((M, K), -1, 1, 5).numpy())
    B = dev(inputs.uniform((K, N), -1, 1, 6).numpy())
    C = unit(A, B)
    n = 64
    cells = torch.empty(2 * n, dtype=torch.int64, device="cuda")
    bsg.audit(A, B, C, seed=7, nsamples=n, cells=cells)
    pairs = [tuple(p) for p in cells.cpu().numpy().reshape(n, 2)]
    i, j = pairs[0]
    Cv = C.view(torch.int32)
    Cv[i, j] ^= 1                     # one bit of one sampled cell
    mis = bsg.audit(A, B, C, seed=7, nsamples=n)
    torch.cuda.synchronize()
    assert int(mis.item()) == pairs.count((i, j)) >= 1


def test_audit_finds_a_wrong_relu_flag():
    M, N, K = 128, 128, 128
    A = dev(inputs.normal((M, K), 1.0, 8).numpy())
    B = dev(inputs.normal((K, N), 1.0, 9).numpy())
    C = unit(A, B, relu=True)
    mis = bsg.audit(A, B, C, relu=False, seed=1, nsamples=512)
    torch.cuda.synchronize()
    assert int(mis.item()) > 0        # about half the cells are negative before the ReLU


def test_audit_skips_rows_with_nonfinite_values():
    M, N, K = 64, 64, 64
    A = inputs.normal((M, K), 1.0, 10).numpy()
    B = inputs.normal((K, N), 1.0, 11).numpy()
    A[:, 5] = np.inf                  # every row holds an Inf: every cell's output is unspecified
    Ad, Bd = dev(A), dev(B)
    C = torch.zeros(M, N, device="cuda")
    mis = bsg.audit(Ad, Bd, C, seed=2, nsamples=256)
    torch.cuda.synchronize()
    assert int(mis.item()) == 0


def test_selftest_passes():
    st, mis, hash_ok = bsg.selftest()
    assert (st, mis, hash_ok) == (0, 0, True)
