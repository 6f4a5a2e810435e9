"""Weight storage (bsg_wquant_cols / bsg_wdequant_cols) against the oracle, bitwise.

Rule: "Precision" manual (docs.presk-lang.org/presk_manual/precision), section
"Integer weights":
- per-column scales of a K x N weight contracted over K, absmax or pow2;
- int8 or int4 codes, with zero channels;
- stored weights f32(q*s).

Parity covers the codes (int4 packed, byte for byte), the scales and the
dequantized weights on ragged shapes with all-zero, underflowing and tie
columns, plus the GPT-2 fc weight at full size, and the non-finite status bit.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal, dev, host
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu


def weights(K, N, seed, std=1.0):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((K, N)) * std).astype(np.float32)
    if N > 3:
        W[:, 0] = 0.0                                       # all-zero channel
        W[:, 1] = np.float32(2.0 ** -149)                   # scale rounds to zero
        # a tie column: pow2 scale 1/2 at 4 bits, entries odd quarters (w/s = k + 1/2)
        col = np.float32([3.0, 1.25, 0.75, -1.25, -0.75, 0.25, -0.25, 1.75])
        W[:, 2] = np.resize(col, K)
    return W


@pytest.mark.parametrize("shape", [(37, 23), (5, 1), (300, 7), (1000, 66), (64, 1), (5000, 77),
                                   (8192, 40), (257, 130)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("pow2", [False, True], ids=["absmax", "pow2"])
def test_codes_scales_and_stored_weights(orc, shape, bits_, pow2):
    K, N = shape
    W = weights(K, N, K * 7 + N + bits_)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q, sc = bsg.wquant_cols(dev(W), bits_, pow2, dstatus=st)
    What = bsg.wdequant_cols(Q, sc, N, bits_)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Qo, so, sto = orc.wquant_cols(W, bits_, pow2)
    assert sto == 0
    assert_bits_equal(host(sc), so, "scales")
    if bits_ == 8:
        assert (host(Q) == Qo).all()
    else:
        assert (host(Q) == orc.pack_int4(Qo)).all()
    assert_bits_equal(host(What), orc.wdequant_cols(Qo, so), "stored weights")


@pytest.mark.parametrize("bits_,pow2", [(8, False), (4, True)])
def test_gpt2_fc_weight_full(orc, bits_, pow2):
    W = inputs.gpt2_weights(768, 3072, 2).numpy()       # the fc weight, N(0, 0.02)
    K, N = W.shape
    Q, sc = bsg.wquant_cols(dev(W), bits_, pow2)
    What = bsg.wdequant_cols(Q, sc, N, bits_)
    torch.cuda.synchronize()
    Qo, so, _ = orc.wquant_cols(W, bits_, pow2)
    assert_bits_equal(host(sc), so, "scales")
    want = Qo if bits_ == 8 else orc.pack_int4(Qo)
    assert (host(Q) == want).all()
    assert_bits_equal(host(What), orc.wdequant_cols(Qo, so), "stored weights")


def test_nonfinite_sets_status():
    W = np.ones((16, 40), np.float32)
    W[3, 37] = np.inf
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsg.wquant_cols(dev(W), 8, False, dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 1


@pytest.mark.parametrize("bits_", [8, 4])
def test_unaligned_weight_rows(orc, bits_):
    """A weight whose rows are not 16-byte aligned (a column slice of a wider
    matrix, ldw = 69): the element-by-element load path, against the oracle."""
    K, N, ldw = 600, 66, 69
    Wfull = weights(K, ldw, 11 + bits_)
    Wd = dev(Wfull)
    width = N if bits_ == 8 else (N + 1) // 2
    Q = torch.zeros((K, width), dtype=torch.int8 if bits_ == 8 else torch.uint8, device="cuda")
    sc = torch.zeros(N, dtype=torch.float32, device="cuda")
    import ctypes
    rc = bsg.load().bsg_wquant_cols(ctypes.c_void_p(Wd.data_ptr()), K, N, ldw, bits_, 0,
                                    ctypes.c_void_p(Q.data_ptr()), width,
                                    ctypes.c_void_p(sc.data_ptr()), None, None)
    assert rc == 0
    torch.cuda.synchronize()
    Qo, so, _ = orc.wquant_cols(np.ascontiguousarray(Wfull[:, :N]), bits_, False)
    assert_bits_equal(host(sc), so, "scales")
    want = Qo if bits_ == 8 else orc.pack_int4(Qo)
    assert (host(Q) == want).all()
