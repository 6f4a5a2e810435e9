"""Weight storage (bsg_wquant_cols / bsg_wdequant_cols) against the oracle, bitwise.

Rule: "Precision" manual (docs.presk-lang.org/presk_manual/precision), section
"Integer weights":
- per-column scales of a K x N weight contracted over K, absmax or pow2;
- int8 or int4 codes, with zero channels;
- stored weights f32(q*s).

Parity covers the codes (int4 packed, byte for byte), the scales and the
dequantized weights on ragged shapes with all-zero, underflowing, subnormal
and tie columns, plus the GPT-2 fc weight at full size, and the non-finite status bit.
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
    if N > 4:
        # subnormal entries: a scale near 2^-137, whose f32 reciprocal
        # overflows to +Inf, so every code takes the kernels' exact path
        W[:, 3] = (rng.standard_normal(K) * 2.0 ** -130).astype(np.float32)
    return W


@pytest.mark.parametrize("path", ["", "cluster", "lag"])
@pytest.mark.parametrize("shape", [(37, 23), (5, 1), (300, 7), (1000, 66), (64, 1), (5000, 77),
                                   (8192, 40), (257, 130), (6000, 300)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("bits_", [8, 4])
@pytest.mark.parametrize("pow2", [False, True], ids=["absmax", "pow2"])
def test_codes_scales_and_stored_weights(orc, monkeypatch, path, shape, bits_, pow2):
    """Each path (the cluster kernel, the one-read item list of long columns,
    and the default choice between them) on every shape."""
    monkeypatch.setenv("BSG_WQ_PATH", path)
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


@pytest.mark.parametrize("path", ["cluster", "lag"])
@pytest.mark.parametrize("bits_", [8, 4])
def test_quotients_near_half_integers(orc, monkeypatch, path, bits_):
    """Columns whose scale is exactly 1 (max |w| = 2^(b-1) - 1) and whose
    entries sit a hair from half-integers -- 2^-16 to 2^-12 above and below,
    and exactly on them -- so that the codes straddle the kernels' fast test
    (the product with the reciprocal scale more than 2^-14 from a
    half-integer) and its exact fallback: codes bitwise the oracle's."""
    monkeypatch.setenv("BSG_WQ_PATH", path)
    qmax = 127 if bits_ == 8 else 7
    deltas = [0.0] + [sg * 2.0 ** -e for e in (12, 13, 14, 15, 16) for sg in (1, -1)]
    base = [0.5, 1.5, 2.5, 3.5, -0.5, -2.5, 5.5 if bits_ == 4 else 100.5]
    vals = [np.float32(b + d) for b in base for d in deltas]
    K = 5000
    W = np.zeros((K, 6), np.float32)
    for j in range(6):
        W[:, j] = np.resize(np.float32(vals[j::1]), K)
        W[7 * j, j] = np.float32(qmax)          # max |w| = qmax: s = 1
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q, sc = bsg.wquant_cols(dev(W), bits_, False, dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Qo, so, _ = orc.wquant_cols(W, bits_, False)
    assert (so == 1.0).all()
    assert_bits_equal(host(sc), so, "scales")
    want = Qo if bits_ == 8 else orc.pack_int4(Qo)
    assert (host(Q) == want).all()


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


@pytest.mark.parametrize("K", [16, 5000])
def test_nonfinite_sets_status(K):
    W = np.ones((K, 40), np.float32)
    W[3, 37] = np.inf
    W[K - 1, 2] = np.nan
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsg.wquant_cols(dev(W), 8, False, dstatus=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 1
    assert not int(st.item()) & 2, "a bounded wait expired"


@pytest.mark.parametrize("K", [600, 5000])
@pytest.mark.parametrize("bits_", [8, 4])
def test_unaligned_weight_rows(orc, bits_, K):
    """A weight whose rows are not 16-byte aligned (a column slice of a wider
    matrix, ldw = 69): the element-by-element loads of the cluster kernel and
    the one-read path's scalar loads, against the oracle."""
    N, ldw = 66, 69
    Wfull = weights(K, ldw, 11 + bits_)
    Wd = dev(Wfull)
    width = N if bits_ == 8 else (N + 1) // 2
    Q = torch.zeros((K, width), dtype=torch.int8 if bits_ == 8 else torch.uint8, device="cuda")
    sc = torch.zeros(N, dtype=torch.float32, device="cuda")
    import ctypes
    lib = bsg.load()
    nws = lib.bsg_wquant_cols_workspace_size(K, N)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    rc = lib.bsg_wquant_cols(ctypes.c_void_p(Wd.data_ptr()), K, N, ldw, bits_, 0,
                             ctypes.c_void_p(Q.data_ptr()), width, ctypes.c_void_p(sc.data_ptr()),
                             ctypes.c_void_p(ws.data_ptr()), nws, None, None)
    assert rc == 0
    torch.cuda.synchronize()
    Qo, so, _ = orc.wquant_cols(np.ascontiguousarray(Wfull[:, :N]), bits_, False)
    assert_bits_equal(host(sc), so, "scales")
    want = Qo if bits_ == 8 else orc.pack_int4(Qo)
    assert (host(Q) == want).all()
