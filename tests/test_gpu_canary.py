"""Out-of-bounds writes: every output and every workspace is surrounded by
canary bytes, and after each call the canaries must be intact while the
outputs are bitwise the oracle's.

Covers the ragged edges where a store could run past its region: C with a
leading dimension larger than N (aligned, so stored through TMA, and
unaligned, so stored with plain stores), rows of C past M, the int8 codes
and scale arrays of the quantize entry points, the chained units' outputs,
the packed int4 weight codes, and the tail of each workspace past the size
its *_workspace_size function reports.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal, host
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu

CANARY_F32 = 0x7FC0DEAD          # a NaN bit pattern no kernel produces
CANARY_BYTE = 0xA5
TAIL = 4096                      # canary bytes after each workspace


def lib():
    return bsg.load()


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def canary_f32(n):
    return torch.full((n,), CANARY_F32, dtype=torch.int32, device="cuda").view(torch.float32)


def workspace(nbytes):
    """A device buffer of nbytes + TAIL canary bytes; returns (tensor, ptr)."""
    buf = torch.full((nbytes + TAIL + 256,), CANARY_BYTE, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    return buf, off


def tail_intact(buf, off, nbytes):
    t = host(buf[off + nbytes: off + nbytes + TAIL])
    return bool((t == CANARY_BYTE).all())


def ptr(t, byte_off=0):
    return ctypes.c_void_p(t.data_ptr() + byte_off)


@pytest.mark.parametrize("M,N,K,extra", [(300, 150, 200, 1), (300, 152, 200, 4),
                                         (257, 1025, 1100, 3), (129, 256, 64, 8),
                                         (1, 1, 1, 1), (640, 300, 4097, 5)],
                         ids=lambda v: str(v))
def test_gemm_writes_only_its_c(orc, M, N, K, extra):
    """C in a buffer with ldc = N + extra (extra = 4, 8: rows 16-byte aligned,
    TMA stores; otherwise plain stores) and two spare rows: the padding
    columns, the spare rows and the workspace tail keep their canaries."""
    A = inputs.normal((M, K), 1.0, M + K).numpy()
    B = inputs.adversarial(N, K, N + K, along_rows=False).numpy()
    ldc = N + extra
    C = canary_f32((M + 2) * ldc)
    nws = lib().bsgemm_i8_workspace_size(M, N, K)
    ws, off = workspace(nws)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    rc = lib().bsgemm_i8_ex(ptr(Ad), K, 0, ptr(Bd), N, 0, M, N, K, 1, ptr(C), ldc,
                            ptr(ws, off), nws, ptr(st), stream())
    assert rc == 0
    torch.cuda.synchronize()
    Ch = host(C).reshape(M + 2, ldc)
    Co, _ = orc.bsgemm_i8(A, B, True)
    assert_bits_equal(np.ascontiguousarray(Ch[:M, :N]), Co, "C")
    assert (Ch[:M, N:].view(np.uint32) == CANARY_F32).all(), "padding columns written"
    assert (Ch[M:].view(np.uint32) == CANARY_F32).all(), "rows past M written"
    assert tail_intact(ws, off, nws), "workspace tail written"


@pytest.mark.parametrize("rows,cols,extra", [(37, 100, 3), (5000, 70, 2), (300, 33, 4)],
                         ids=lambda v: str(v))
def test_quantize_entry_points_write_only_their_outputs(orc, rows, cols, extra):
    X = inputs.adversarial(rows, cols, rows + cols).numpy()
    Xd = torch.from_numpy(X).cuda()
    ldq = cols + extra
    # rows: codes rows x ldq, scale and inv with 8 spare floats each
    Q = torch.full(((rows + 1) * ldq,), -86, dtype=torch.int8, device="cuda")   # 0xAA
    sc, iv = canary_f32(rows + 8), canary_f32(rows + 8)
    assert lib().bsg_quantize_rows(ptr(Xd), rows, cols, cols, ptr(Q), ldq, ptr(sc), ptr(iv),
                                   None, stream()) == 0
    torch.cuda.synchronize()
    Qh = host(Q).reshape(rows + 1, ldq)
    Qo, sco, ivo, _ = orc.quantize_rows(X)
    assert_bits_equal(np.ascontiguousarray(Qh[:rows, :cols]), Qo, "row codes")
    assert (Qh[:rows, cols:] == -86).all() and (Qh[rows:] == -86).all()
    assert_bits_equal(host(sc)[:rows], sco, "row scales")
    assert (host(sc)[rows:].view(np.uint32) == CANARY_F32).all()
    assert (host(iv)[rows:].view(np.uint32) == CANARY_F32).all()
    # columns: the same layout, a scale per column, and a canaried workspace
    Q = torch.full(((rows + 1) * ldq,), -86, dtype=torch.int8, device="cuda")
    sc, iv = canary_f32(cols + 8), canary_f32(cols + 8)
    nws = lib().bsg_quantize_cols_workspace_size(rows, cols)
    ws, off = workspace(nws)
    assert lib().bsg_quantize_cols(ptr(Xd), rows, cols, cols, ptr(Q), ldq, ptr(sc), ptr(iv),
                                   ptr(ws, off), nws, None, stream()) == 0
    torch.cuda.synchronize()
    Qh = host(Q).reshape(rows + 1, ldq)
    Qo, sco, ivo, _ = orc.quantize_cols(X)
    assert_bits_equal(np.ascontiguousarray(Qh[:rows, :cols]), Qo, "column codes")
    assert (Qh[:rows, cols:] == -86).all() and (Qh[rows:] == -86).all()
    assert_bits_equal(host(iv)[:cols], ivo, "column inv")
    assert (host(sc)[cols:].view(np.uint32) == CANARY_F32).all()
    assert tail_intact(ws, off, nws)


def test_chained_units_write_only_their_outputs(orc):
    M, K, N1, N2 = 333, 130, 517, 75
    A = inputs.normal((M, K), 1.0, 5).numpy()
    B1 = inputs.normal((K, N1), 0.1, 6).numpy()
    B2 = inputs.normal((N1, N2), 0.1, 7).numpy()
    Ad, B1d, B2d = (torch.from_numpy(x).cuda() for x in (A, B1, B2))
    # requant: C, codes, scales and inv each followed by canaries
    C = canary_f32(M * N1 + 64)
    Cq = torch.full((M * N1 + 64,), -86, dtype=torch.int8, device="cuda")
    sc, iv = canary_f32(M + 8), canary_f32(M + 8)
    nws = lib().bsgemm_i8_requant_workspace_size(M, N1, K)
    ws, off = workspace(nws)
    assert lib().bsgemm_i8_requant(ptr(Ad), ptr(B1d), M, N1, K, 1, ptr(C), ptr(Cq), ptr(sc),
                                   ptr(iv), ptr(ws, off), nws, None, stream()) == 0
    torch.cuda.synchronize()
    Co, _ = orc.bsgemm_i8(A, B1, True)
    Qo, sco, _, _ = orc.quantize_rows(Co)
    assert_bits_equal(host(C)[:M * N1].reshape(M, N1), Co, "requant C")
    assert_bits_equal(host(Cq)[:M * N1].reshape(M, N1), Qo, "requant codes")
    assert_bits_equal(host(sc)[:M], sco, "requant scales")
    assert (host(C)[M * N1:].view(np.uint32) == CANARY_F32).all()
    assert (host(Cq)[M * N1:] == -86).all()
    assert (host(sc)[M:].view(np.uint32) == CANARY_F32).all()
    assert (host(iv)[M:].view(np.uint32) == CANARY_F32).all()
    assert tail_intact(ws, off, nws)
    # chain: C1, C2 followed by canaries
    C1, C2 = canary_f32(M * N1 + 64), canary_f32(M * N2 + 64)
    nws = lib().bsgemm_i8_chain_workspace_size(M, K, N1, N2)
    ws, off = workspace(nws)
    assert lib().bsgemm_i8_chain(ptr(Ad), ptr(B1d), ptr(B2d), M, K, N1, N2, 1, 0, ptr(C1),
                                 ptr(C2), ptr(ws, off), nws, None, stream()) == 0
    torch.cuda.synchronize()
    C2o, _ = orc.bsgemm_i8(Co, B2, False)
    assert_bits_equal(host(C1)[:M * N1].reshape(M, N1), Co, "chain C1")
    assert_bits_equal(host(C2)[:M * N2].reshape(M, N2), C2o, "chain C2")
    assert (host(C1)[M * N1:].view(np.uint32) == CANARY_F32).all()
    assert (host(C2)[M * N2:].view(np.uint32) == CANARY_F32).all()
    assert tail_intact(ws, off, nws)


@pytest.mark.parametrize("K", [77, 5000])
@pytest.mark.parametrize("bits", [8, 4])
def test_weight_storage_writes_only_its_codes(orc, bits, K):
    N = 41
    W = inputs.normal((K, N), 0.02, 9).numpy()
    Wd = torch.from_numpy(W).cuda()
    width = N if bits == 8 else (N + 1) // 2
    ldq = width + 3
    Q = torch.full(((K + 1) * ldq,), -86, dtype=torch.int8, device="cuda")
    sc = canary_f32(N + 8)
    nws = lib().bsg_wquant_cols_workspace_size(K, N)
    ws, off = workspace(nws)
    assert lib().bsg_wquant_cols(ptr(Wd), K, N, N, bits, 0, ptr(Q), ldq, ptr(sc), ptr(ws, off),
                                 nws, None, stream()) == 0
    torch.cuda.synchronize()
    Qh = host(Q).reshape(K + 1, ldq)
    Qo, sco, _ = orc.wquant_cols(W, bits=bits)
    got = np.ascontiguousarray(Qh[:K, :width])
    if bits == 4:
        Qo = orc.pack_int4(Qo)
        got = got.view(np.uint8)
    assert_bits_equal(got, Qo, "codes")
    assert (Qh[:K, width:] == -86).all() and (Qh[K:] == -86).all()
    assert_bits_equal(host(sc)[:N], sco, "scales")
    assert (host(sc)[N:].view(np.uint32) == CANARY_F32).all()
    assert tail_intact(ws, off, nws)


@pytest.mark.parametrize("M,N,K,extra", [(257, 1025, 1100, 3), (130, 96, 2100, 4)],
                         ids=lambda v: str(v))
def test_int32_accumulators_write_only_their_s(orc, M, N, K, extra):
    """bsg_gemm_s32 (the contraction with int32 S stored) into a padded S."""
    rng = np.random.default_rng(M + N + K)
    Aq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    Bq = rng.integers(-127, 128, (K, N)).astype(np.int8)
    Ad, Bd = torch.from_numpy(Aq).cuda(), torch.from_numpy(Bq).cuda()
    lds = N + extra
    S = torch.full(((M + 2) * lds,), CANARY_F32, dtype=torch.int32, device="cuda")
    nws = lib().bsg_gemm_s32_workspace_size(M, N, K)
    ws, off = workspace(nws)
    assert lib().bsg_gemm_s32(ptr(Ad), K, ptr(Bd), N, M, N, K, ptr(S), lds, ptr(ws, off), nws,
                              None, stream()) == 0
    torch.cuda.synchronize()
    Sh = host(S).reshape(M + 2, lds)
    So, _ = orc.gemm_s32(Aq, Bq)
    assert_bits_equal(np.ascontiguousarray(Sh[:M, :N]), So, "S")
    assert (Sh[:M, N:] == CANARY_F32).all() and (Sh[M:] == CANARY_F32).all()
    assert tail_intact(ws, off, nws)


def test_grouped_launch_writes_only_its_cs(orc):
    """Three units in one launch, each C padded differently."""
    shapes = [(300, 150, 200, 1), (257, 1025, 1100, 3), (129, 96, 700, 4)]
    items = (bsg.GemmItem * 3)()
    keep, want = [], []
    for i, (M, N, K, extra) in enumerate(shapes):
        A = inputs.normal((M, K), 1.0, 40 + i).numpy()
        B = inputs.normal((K, N), 0.1, 50 + i).numpy()
        Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        ldc = N + extra
        C = canary_f32((M + 2) * ldc)
        nws = lib().bsgemm_i8_workspace_size(M, N, K)
        ws, off = workspace(nws)
        items[i] = bsg.GemmItem(Ad.data_ptr(), K, 0, Bd.data_ptr(), N, 0, M, N, K, i % 2,
                                C.data_ptr(), ldc, ws.data_ptr() + off, nws)
        keep.append((Ad, Bd, C, ws, off, nws, M, N, ldc))
        want.append(orc.bsgemm_i8(A, B, bool(i % 2))[0])
    assert lib().bsgemm_i8_group(items, 3, None, stream()) == 0
    torch.cuda.synchronize()
    for (Ad, Bd, C, ws, off, nws, M, N, ldc), Co in zip(keep, want):
        Ch = host(C).reshape(M + 2, ldc)
        assert_bits_equal(np.ascontiguousarray(Ch[:M, :N]), Co, f"group C {M}x{N}")
        assert (Ch[:M, N:].view(np.uint32) == CANARY_F32).all()
        assert (Ch[M:].view(np.uint32) == CANARY_F32).all()
        assert tail_intact(ws, off, nws)


def test_host_entry_point_writes_only_its_c(orc):
    """bsgemm_i8_host: C on the host followed by canaries, and the device
    workspace's tail."""
    M, N, K = 700, 333, 900
    A = inputs.normal((M, K), 1.0, 61)
    B = inputs.normal((K, N), 0.1, 62)
    Ah, Bh = A.pin_memory(), B.pin_memory()
    C = torch.full((M * N + 64,), CANARY_F32, dtype=torch.int32).view(torch.float32).pin_memory()
    nws = lib().bsgemm_i8_host_workspace_size(M, N, K)
    ws, off = workspace(nws)
    st = ctypes.c_int32(-1)
    assert lib().bsgemm_i8_host(ptr(Ah), ptr(Bh), M, N, K, 0, ptr(C), ptr(ws, off), nws,
                                ctypes.byref(st), stream()) == 0
    assert st.value == 0
    Co, _ = orc.bsgemm_i8(A.numpy(), B.numpy(), False)
    Cn = C.numpy()
    assert_bits_equal(Cn[:M * N].reshape(M, N), Co, "host C")
    assert (Cn[M * N:].view(np.uint32) == CANARY_F32).all()
    assert tail_intact(ws, off, nws)
