"""Several units in one GEMM launch (bsgemm_i8_group) against the oracle and
against the one-at-a-time entry point, bitwise.

Rule: "Verification -- why you can trust the numbers", section "The verified
INT8 units": each product is defined by its own operands, so sharing a launch
(and its tiles) with other products must not change a bit of it.

Cases:
- ragged items with transposes and ReLU;
- an item with M <= 128 beside large ones;
- every kernel forced;
- the training trio at full size, grouped, against bsgemm_i8_ex.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal, dev, host
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu


def stored(M, N, K, tA, tB, seed):
    A = inputs.normal((K, M) if tA else (M, K), 1.0, seed).numpy()
    B = inputs.normal((N, K) if tB else (K, N), 1.0, seed + 1).numpy()
    Am = np.ascontiguousarray(A.T) if tA else A
    Bm = np.ascontiguousarray(B.T) if tB else B
    return A, B, Am, Bm


GROUPS = [
    [(300, 200, 100, False, False, True), (129, 257, 1025, True, False, False),
     (520, 383, 2100, False, True, True)],
    [(64, 500, 700, False, False, False), (1000, 66, 300, False, False, True)],
    [(257, 129, 64, True, True, False)],
]


@pytest.mark.parametrize("gi", range(len(GROUPS)))
def test_group_matches_oracle(orc, gi):
    items, want = [], []
    for i, (M, N, K, tA, tB, relu) in enumerate(GROUPS[gi]):
        A, B, Am, Bm = stored(M, N, K, tA, tB, 100 * gi + 10 * i)
        items.append((dev(A), dev(B), tA, tB, relu))
        want.append(orc.bsgemm_i8(Am, Bm, relu)[0])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = bsg.bsgemm_i8_group(items, dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i, (C, Co) in enumerate(zip(outs, want)):
        assert_bits_equal(host(C), Co, f"group {gi} item {i}")


@pytest.mark.parametrize("bn", [64, 128, 192, 256])
@pytest.mark.parametrize("pair", [True, False], ids=["pair", "single"])
def test_group_every_kernel(orc, monkeypatch, bn, pair):
    monkeypatch.setenv("BSG_GEMM_BN", str(bn))
    monkeypatch.setenv("BSG_GEMM_PAIR", "1" if pair else "0")
    items, want = [], []
    for i, (M, N, K, tA, tB, relu) in enumerate(GROUPS[0]):
        A, B, Am, Bm = stored(M, N, K, tA, tB, 7 + i)
        items.append((dev(A), dev(B), tA, tB, relu))
        want.append(orc.bsgemm_i8(Am, Bm, relu)[0])
    outs = bsg.bsgemm_i8_group(items)
    torch.cuda.synchronize()
    for i, (C, Co) in enumerate(zip(outs, want)):
        assert_bits_equal(host(C), Co, f"bn={bn} pair={pair} item {i}")


def test_training_trio_grouped_equals_one_at_a_time():
    X, W, dY = (dev(t.numpy()) for t in inputs.train_trio())
    ops = [(X, W, False, False, False),        # forward X.W
           (dY, W, False, True, False),        # grad-input dY.W^T (W stored K x N = N' x K')
           (X, dY, True, False, False)]        # grad-weight X^T.dY
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    grouped = bsg.bsgemm_i8_group(ops, dstatus=st)
    single = [bsg.bsgemm_i8_ex(A, B, transA=tA, transB=tB, relu=r) for A, B, tA, tB, r in ops]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for name, g, s in zip(("fwd", "dgrad", "wgrad"), grouped, single):
        assert_bits_equal(host(g), host(s), name)
