"""GPU parity of the chained units against the oracle's composition, bitwise.

Rule: the B2B chain of "Verification -- why you can trust the numbers",
section "Layer 1: exact init gates" (one unit's output feeds the next), and
the W8A8 requantisation of the presk "Precision" manual's closing list.  The
oracle needs no arithmetic of its own here: bsgemm_i8_requant must equal
quantize_rows(bsgemm_i8(A, B)) and bsgemm_i8_chain must equal
bsgemm_i8(bsgemm_i8(A, B1), B2), both computed by the oracle.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal, dev, host
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu


def requant(A, B, relu):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C, Cq, sc, iv = bsg.bsgemm_i8_requant(dev(A), dev(B), relu=relu, dstatus=st)
    torch.cuda.synchronize()
    return host(C), host(Cq), host(sc), host(iv), int(st.item())


def check_requant(orc, A, B, relu, what, rows=None):
    C, Cq, sc, iv, st = requant(A, B, relu)
    Co, _ = orc.bsgemm_i8(A, B, relu)
    assert_bits_equal(C, Co, what + " C")
    Qo, sco, ivo, _ = orc.quantize_rows(Co)
    r = slice(None) if rows is None else rows
    assert_bits_equal(Cq[r], Qo[r], what + " codes")
    assert_bits_equal(sc[r], sco[r], what + " scales")
    assert_bits_equal(iv[r], ivo[r], what + " inv")
    return C, st


@pytest.mark.parametrize("shape,relu", [((1, 1, 1), False), ((300, 150, 200), True),
                                        ((257, 2049, 1100), False), ((128, 20000, 768), True),
                                        ((1000, 333, 64), False)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_requant_matches_oracle_composition(orc, shape, relu):
    M, N, K = shape
    A = inputs.normal((M, K), 1.0, M + 7)
    B = inputs.normal((K, N), 0.05, N + 11)
    _, st = check_requant(orc, A.numpy(), B.numpy(), relu, f"{shape}")
    assert st == 0


def test_requant_gpt2_fc_full(orc):
    A, B, relu = inputs.gpt2_linear_inputs("fc")
    _, st = check_requant(orc, A.numpy(), B.numpy(), relu, "fc")
    assert st == 0


def test_requant_overflowed_rows_set_nonfinite(orc):
    """Adversarial A rows of magnitude 1e30 times B columns of 1e30 overflow C
    to +-Inf: those rows set the non-finite bit (their codes are then
    unspecified); every other row is bitwise the oracle's."""
    A = inputs.adversarial(300, 200, 12).numpy()
    B = inputs.adversarial(150, 200, 13, along_rows=False).numpy()
    Co, _ = orc.bsgemm_i8(A, B)
    finite = np.isfinite(Co).all(axis=1)
    assert (~finite).any() and finite.any()
    C, st = check_requant(orc, A, B, False, "adversarial", rows=finite)
    assert st & 1


@pytest.mark.parametrize("case", ["gpt2_mlp", "ragged", "wide", "deep"])
def test_chain_matches_two_units(orc, case):
    if case == "gpt2_mlp":
        # the GPT-2-small MLP at M = 8192: fc (768 -> 3072, ReLU) then proj
        A = inputs.gpt2_activations(8192, 768, 2)
        B1 = inputs.gpt2_weights(768, 3072, 2)
        B2 = inputs.gpt2_weights(3072, 768, 3)
        relu1, relu2 = True, False
    elif case == "ragged":
        A = inputs.normal((333, 130), 1.0, 5)
        B1 = inputs.normal((130, 517), 0.1, 6)
        B2 = inputs.normal((517, 75), 0.1, 7)
        relu1, relu2 = False, True
    elif case == "deep":
        # K > 2048: the first unit quantizes B1 on the second stream too
        A = inputs.normal((130, 3000), 1.0, 11)
        B1 = inputs.normal((3000, 700), 0.05, 12)
        B2 = inputs.normal((700, 64), 0.05, 13)
        relu1, relu2 = True, True
    else:
        A = inputs.normal((256, 512), 1.0, 8)
        B1 = inputs.normal((512, 5000), 0.05, 9)
        B2 = inputs.normal((5000, 384), 0.05, 10)
        relu1, relu2 = True, False
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    C1, C2 = bsg.bsgemm_i8_chain(dev(A), dev(B1), dev(B2), relu1, relu2, dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    C1o, _ = orc.bsgemm_i8(A.numpy(), B1.numpy(), relu1)
    C2o, _ = orc.bsgemm_i8(C1o, B2.numpy(), relu2)
    assert_bits_equal(host(C1), C1o, case + " C1")
    assert_bits_equal(host(C2), C2o, case + " C2")
    # and the same as two separate units on the GPU
    C2s = bsg.bsgemm_i8(bsg.bsgemm_i8(dev(A), dev(B1), relu=relu1), dev(B2), relu=relu2)
    assert_bits_equal(host(C2), host(C2s), case + " C2 vs two units")


def _tie_inputs(M=64, N=96, seed=3):
    """A = 127 I (row scales 1) and B with a row of 127 (column scales 1) and
    rows of odd values +-1 holding one +-2: the first unit's C is exactly
    127 B, so each C row below the first has max 254 (scale 2, inv 1/2) and
    its odd entries quantize from x * inv = +-63.5, exact ties."""
    rng = np.random.default_rng(seed)
    A = (127.0 * np.eye(M)).astype(np.float32)
    B = rng.choice([-1.0, 1.0], size=(M, N)).astype(np.float32)
    B[0, :] = 127.0
    for i in range(1, M):
        B[i, rng.integers(0, N)] = 2.0 * rng.choice([-1.0, 1.0])
    return A, B


def test_chain_gate_hunts_quantize_ties(orc):
    """The chain gate of "Layer 1: exact init gates": inputs on which the
    spec's floor(x*inv + 0.5) and round-half-to-even disagree in the second
    unit's quantize, so that agreeing with the oracle is not vacuous."""
    A, B = _tie_inputs()
    C, Cq, sc, _, st = requant(A, B, False)
    assert st == 0
    Co, _ = orc.bsgemm_i8(A, B, False)
    assert_bits_equal(C, (127.0 * B).astype(np.float32), "C = 127 B exactly")
    Qo, sco, _, _ = orc.quantize_rows(Co)
    assert_bits_equal(Cq, Qo, "codes follow the spec")
    assert (sc[1:] == 2.0).all()
    # the round-half-to-even reading differs on every -63.5
    rne = np.rint(C[1:] * 0.5).astype(np.int8)
    disagree = (rne != Qo[1:]).sum()
    assert disagree > 0 and (Cq[1:][C[1:] == -127.0] == -63).all()
    # the chained second unit inherits the tie rule: C2 = 2 * (q(C1) . B2)
    B2 = np.zeros((B.shape[1], 8), np.float32)
    B2[np.arange(8), np.arange(8)] = 127.0
    Cd1, Cd2 = bsg.bsgemm_i8_chain(dev(A), dev(B), dev(B2))
    torch.cuda.synchronize()
    C2o, _ = orc.bsgemm_i8(Co, B2, False)
    assert_bits_equal(host(Cd2), C2o, "chain C2")
    assert (host(Cd2)[1:] != (2.0 * 127.0 * rne[:, :8]).astype(np.float32)).any()
