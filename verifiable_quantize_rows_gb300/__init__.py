"""Bit-exact block-scaled int8 GEMM for GB300 (sm_103a).

A thin Python binding over the C ABI declared in ``include/bsgemm.h``
(library ``_build/libbsgemm.so``).  Every step of the computation runs in the
library's CUDA kernels; this module only checks and marshals arguments, and
uses PyTorch for device memory and streams.  There is no CPU fallback: if the
library is missing or the device is not sm_103, calls raise.

Functions take contiguous row-major CUDA tensors and run on the current
PyTorch stream (or the ``stream`` given).

Workspaces: a call given no ``workspace`` uses one buffer per device shared
by every such call.  Calls that may run at the same time (on different
streams, or from different host threads) must each pass their own
``Workspace``, and so should calls on a stream other than PyTorch's current
one: when the shared buffer grows, the old one goes back to PyTorch's
allocator, which tracks only the stream it was allocated on.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

__all__ = ["BsgError", "load", "exported_symbols", "quantize_rows", "quantize_cols",
           "gemm_s32", "epilogue", "bsgemm_i8", "bsgemm_i8_ex", "bsgemm_i8_host",
           "bsgemm_i8_quantize", "bsgemm_i8_contract", "launch_count", "selftest_scales", "gemm_tile_width", "hash_f32", "probe_hash", "probe_hash_async", "workspace_size", "Workspace",
           "DSTATUS_NONFINITE", "DSTATUS_TIMEOUT", "MAX_K"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libbsgemm.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "bsgemm.h")

MAX_K = 133144
DSTATUS_NONFINITE = 0x1
DSTATUS_TIMEOUT = 0x2

STATUS = {0: "BSG_OK", 1: "BSG_ERR_ARG", 2: "BSG_ERR_K_TOO_LARGE", 3: "BSG_ERR_WORKSPACE",
          4: "BSG_ERR_CUDA", 5: "BSG_ERR_NONFINITE", 6: "BSG_ERR_TIMEOUT",
          7: "BSG_ERR_UNSUPPORTED"}


class BsgError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


_lock = threading.Lock()
_lib = None

_i64, _vp, _sz, _i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int


class GemmItem(ctypes.Structure):
    """One item of bsgemm_i8_group (the C struct bsg_gemm_item)."""
    _fields_ = [("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("transA", ctypes.c_int),
                ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("transB", ctypes.c_int),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("relu", ctypes.c_int), ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("workspace", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


class HostItem(ctypes.Structure):
    """One item of bsgemm_i8_host_batch (the C struct bsg_host_item)."""
    _fields_ = [("A_host", ctypes.c_void_p), ("B_host", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("relu", ctypes.c_int), ("C_host", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


def _declare(lib):
    sigs = {
        "bsg_status_str": ([_i32], ctypes.c_char_p),
        "bsg_version": ([], _i32),
        "bsg_quantize_rows": ([_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _vp], _i32),
        "bsg_quantize_cols_workspace_size": ([_i64, _i64], _sz),
        "bsg_quantize_cols": ([_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _sz, _vp, _vp],
                              _i32),
        "bsg_gemm_s32_workspace_size": ([_i64, _i64, _i64], _sz),
        "bsg_gemm_s32": ([_vp, _i64, _vp, _i64, _i64, _i64, _i64, _vp, _i64, _vp, _sz, _vp, _vp],
                         _i32),
        "bsg_epilogue": ([_vp, _i64, _vp, _vp, _i64, _i64, _i32, _vp, _i64, _vp], _i32),
        "bsgemm_i8_workspace_size": ([_i64, _i64, _i64], _sz),
        "bsgemm_i8": ([_vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _sz, _vp, _vp], _i32),
        "bsgemm_i8_ex": ([_vp, _i64, _i32, _vp, _i64, _i32, _i64, _i64, _i64, _i32, _vp, _i64,
                          _vp, _sz, _vp, _vp], _i32),
        "bsgemm_i8_quantize": ([_vp, _i64, _i32, _vp, _i64, _i32, _i64, _i64, _i64, _vp, _sz, _vp,
                                _vp], _i32),
        "bsgemm_i8_contract": ([_i64, _i64, _i64, _i32, _vp, _i64, _vp, _sz, _vp, _vp], _i32),
        "bsg_launch_count": ([], ctypes.c_uint64),
        "bsg_gemm_tile_width": ([_i64, _i64, _i32], _i32),
        "bsg_selftest_scales": ([ctypes.c_uint32, ctypes.c_uint32, _vp], _i32),
        "bsgemm_i8_host_workspace_size": ([_i64, _i64, _i64], _sz),
        "bsgemm_i8_host": ([_vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _sz, _vp, _vp], _i32),
        "bsgemm_i8_host_batch": ([ctypes.POINTER(HostItem), _i32, _vp, _vp], _i32),
        "bsg_hash_f32_workspace_size": ([_i64, _i64], _sz),
        "bsg_hash_f32": ([_vp, _i64, _i64, _i64, _vp, _vp, _sz, _vp], _i32),
        "bsg_probe_workspace_size": ([_i64, _i64, _i64], _sz),
        "bsg_probe_hash_async": ([ctypes.c_uint64, _i64, _i64, _i64, _vp, _vp, _sz, _vp, _vp],
                                 _i32),
        "bsg_probe_hash": ([ctypes.c_uint64, _i64, _i64, _i64, _vp, _vp, _sz, _vp], _i32),
        "bsg_audit": ([_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _i64, _i32, ctypes.c_uint64,
                       _i32, _vp, _vp, _vp], _i32),
        "bsg_selftest_workspace_size": ([], _sz),
        "bsg_selftest": ([_vp, _sz, _vp, _vp], _i32),
        "bsgemm_i8_group": ([ctypes.POINTER(GemmItem), _i32, _vp, _vp], _i32),
        "bsg_wquant_cols_workspace_size": ([_i64, _i64], _sz),
        "bsg_wquant_cols": ([_vp, _i64, _i64, _i64, _i32, _i32, _vp, _i64, _vp, _vp, _sz, _vp,
                             _vp], _i32),
        "bsg_wdequant_cols": ([_vp, _i64, _i64, _i64, _i32, _vp, _vp, _i64, _vp], _i32),
        "bsgemm_i8_requant_workspace_size": ([_i64, _i64, _i64], _sz),
        "bsgemm_i8_requant": ([_vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _sz,
                               _vp, _vp], _i32),
        "bsgemm_i8_chain_workspace_size": ([_i64, _i64, _i64, _i64], _sz),
        "bsgemm_i8_chain": ([_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _i32, _vp, _vp, _vp,
                             _sz, _vp, _vp], _i32),
        "bsg_mma_ceiling": ([_i32, _vp, ctypes.POINTER(ctypes.c_double), _vp], _i32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load(path: str | None = None):
    """Load the CUDA library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"CUDA library not built: {p} is missing "
                    "(run `python -m verifiable_quantize_rows_gb300.build`)")
            lib = _declare(ctypes.CDLL(p))
            if path is not None:
                return lib
            _lib = lib
        return _lib


def exported_symbols() -> list[str]:
    """Function names declared in include/bsgemm.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:bsg|bsgemm)_\w+)\s*\(", text)))


def _check(code: int, where: str):
    if code != 0:
        raise BsgError(code, where)


# ---------------------------------------------------------------------------
# torch-side helpers (memory and streams only)
def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor of dtype {dtype}")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")


class Workspace:
    """A growable device byte buffer (256-byte aligned, from PyTorch).  One
    per stream of concurrent calls; see the module notes on workspaces."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        torch = _torch()
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device or "cuda")
        return self.buf

    def ptr_size(self, nbytes: int):
        b = self.get(nbytes)
        return ctypes.c_void_p(b.data_ptr()), b.numel()


_default_ws: dict = {}


def _ws(workspace, nbytes):
    torch = _torch()
    if workspace is None:
        dev = torch.cuda.current_device()
        workspace = _default_ws.setdefault(dev, Workspace(torch.device("cuda", dev)))
    return workspace.ptr_size(nbytes)


def workspace_size(M: int, N: int, K: int) -> int:
    return int(load().bsgemm_i8_workspace_size(M, N, K))


# ---------------------------------------------------------------------------
def quantize_rows(X, stream=None, dstatus=None):
    """Per-row int8 quantization: (Q int8, scale f32, inv f32)."""
    torch = _torch()
    _need(X, torch.float32, "X")
    R, C = X.shape
    Q = torch.empty((R, C), dtype=torch.int8, device=X.device)
    sc = torch.empty(R, dtype=torch.float32, device=X.device)
    iv = torch.empty(R, dtype=torch.float32, device=X.device)
    _check(load().bsg_quantize_rows(_ptr(X), R, C, C, _ptr(Q), C, _ptr(sc), _ptr(iv),
                                    _ptr(dstatus), _stream_ptr(stream)), "bsg_quantize_rows")
    return Q, sc, iv


def quantize_cols(X, stream=None, dstatus=None, workspace=None):
    """Per-column int8 quantization (Q keeps X's layout): (Q, scale, inv)."""
    torch = _torch()
    _need(X, torch.float32, "X")
    R, C = X.shape
    lib = load()
    Q = torch.empty((R, C), dtype=torch.int8, device=X.device)
    sc = torch.empty(C, dtype=torch.float32, device=X.device)
    iv = torch.empty(C, dtype=torch.float32, device=X.device)
    wp, wn = _ws(workspace, lib.bsg_quantize_cols_workspace_size(R, C))
    _check(lib.bsg_quantize_cols(_ptr(X), R, C, C, _ptr(Q), C, _ptr(sc), _ptr(iv), wp, wn,
                                 _ptr(dstatus), _stream_ptr(stream)), "bsg_quantize_cols")
    return Q, sc, iv


def gemm_s32(Aq, Bq, stream=None, dstatus=None, workspace=None):
    """Exact int32 S = Aq . Bq on the tensor cores."""
    torch = _torch()
    _need(Aq, torch.int8, "Aq")
    _need(Bq, torch.int8, "Bq")
    M, K = Aq.shape
    K2, N = Bq.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    lib = load()
    S = torch.empty((M, N), dtype=torch.int32, device=Aq.device)
    wp, wn = _ws(workspace, lib.bsg_gemm_s32_workspace_size(M, N, K))
    _check(lib.bsg_gemm_s32(_ptr(Aq), K, _ptr(Bq), N, M, N, K, _ptr(S), N, wp, wn,
                            _ptr(dstatus), _stream_ptr(stream)), "bsg_gemm_s32")
    return S


def epilogue(S, sa, sb, relu: bool = False, stream=None):
    """C = epi(S, sa, sb) (+ReLU) for arbitrary int32 S and float scales."""
    torch = _torch()
    _need(S, torch.int32, "S")
    M, N = S.shape
    if sa.numel() != M or sb.numel() != N:
        raise ValueError("scale lengths do not match S")
    C = torch.empty((M, N), dtype=torch.float32, device=S.device)
    _check(load().bsg_epilogue(_ptr(S), N, _ptr(sa.contiguous()), _ptr(sb.contiguous()), M, N,
                               int(bool(relu)), _ptr(C), N, _stream_ptr(stream)), "bsg_epilogue")
    return C


def bsgemm_i8(A, B, relu: bool = False, out=None, stream=None, dstatus=None, workspace=None):
    """C = epi(q_rows(A) . q_cols(B)) (+ReLU), bit-exact."""
    torch = _torch()
    _need(A, torch.float32, "A")
    _need(B, torch.float32, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    lib = load()
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=A.device)
    wp, wn = _ws(workspace, lib.bsgemm_i8_workspace_size(M, N, K))
    _check(lib.bsgemm_i8(_ptr(A), _ptr(B), M, N, K, int(bool(relu)), _ptr(C), wp, wn,
                         _ptr(dstatus), _stream_ptr(stream)), "bsgemm_i8")
    return C


def bsgemm_i8_requant(A, B, relu: bool = False, stream=None, dstatus=None, workspace=None):
    """(C, Cq, scale, inv): the unit's C and C quantized per row (int8 codes,
    row scales and reciprocals) for the next unit."""
    torch = _torch()
    _need(A, torch.float32, "A")
    _need(B, torch.float32, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    lib = load()
    dev = A.device
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    Cq = torch.empty((M, N), dtype=torch.int8, device=dev)
    scale = torch.empty(M, dtype=torch.float32, device=dev)
    inv = torch.empty(M, dtype=torch.float32, device=dev)
    wp, wn = _ws(workspace, lib.bsgemm_i8_requant_workspace_size(M, N, K))
    _check(lib.bsgemm_i8_requant(_ptr(A), _ptr(B), M, N, K, int(bool(relu)), _ptr(C), _ptr(Cq),
                                 _ptr(scale), _ptr(inv), wp, wn, _ptr(dstatus),
                                 _stream_ptr(stream)), "bsgemm_i8_requant")
    return C, Cq, scale, inv


def bsgemm_i8_chain(A, B1, B2, relu1: bool = False, relu2: bool = False, out1=None, out2=None,
                    stream=None, dstatus=None, workspace=None):
    """(C1, C2) with C1 = bsgemm_i8(A, B1), C2 = bsgemm_i8(C1, B2)."""
    torch = _torch()
    for t, nm in ((A, "A"), (B1, "B1"), (B2, "B2")):
        _need(t, torch.float32, nm)
    M, K = A.shape
    if B1.shape[0] != K or B2.shape[0] != B1.shape[1]:
        raise ValueError("inner dimensions differ")
    N1, N2 = B1.shape[1], B2.shape[1]
    lib = load()
    dev = A.device
    C1 = out1 if out1 is not None else torch.empty((M, N1), dtype=torch.float32, device=dev)
    C2 = out2 if out2 is not None else torch.empty((M, N2), dtype=torch.float32, device=dev)
    wp, wn = _ws(workspace, lib.bsgemm_i8_chain_workspace_size(M, K, N1, N2))
    _check(lib.bsgemm_i8_chain(_ptr(A), _ptr(B1), _ptr(B2), M, K, N1, N2, int(bool(relu1)),
                               int(bool(relu2)), _ptr(C1), _ptr(C2), wp, wn, _ptr(dstatus),
                               _stream_ptr(stream)), "bsgemm_i8_chain")
    return C1, C2


def bsgemm_i8_ex(A, B, transA: bool = False, transB: bool = False, relu: bool = False,
                 out=None, stream=None, dstatus=None, workspace=None):
    """C = epi(q_rows(op(A)) . q_cols(op(B))) with op = transpose when asked."""
    torch = _torch()
    _need(A, torch.float32, "A")
    _need(B, torch.float32, "B")
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    K2, N = (B.shape[1], B.shape[0]) if transB else B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    lib = load()
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=A.device)
    wp, wn = _ws(workspace, lib.bsgemm_i8_workspace_size(M, N, K))
    _check(lib.bsgemm_i8_ex(_ptr(A), A.shape[1], int(bool(transA)), _ptr(B), B.shape[1],
                            int(bool(transB)), M, N, K, int(bool(relu)), _ptr(C), N, wp, wn,
                            _ptr(dstatus), _stream_ptr(stream)), "bsgemm_i8_ex")
    return C


def selftest_scales(first_bits: int = 0, last_bits: int = 0x7F7FFFFF) -> int:
    """Mismatches between the device's f32 scale derivation and its f64
    definition over absmax bit patterns [first_bits, last_bits]."""
    n = ctypes.c_uint64(0)
    _check(load().bsg_selftest_scales(first_bits, last_bits, ctypes.byref(n)),
           "bsg_selftest_scales")
    return int(n.value)


def gemm_tile_width(M: int, N: int, sms: int) -> int:
    """Output tile width the GEMM kernel picks for an M x N problem."""
    return int(load().bsg_gemm_tile_width(M, N, sms))


def mma_ceiling(iters: int, stream=None, dstatus=None) -> float:
    """Launch the tensor-pipe ceiling kernel (asynchronous); returns the
    floating-point operations that launch performs."""
    flops = ctypes.c_double(0.0)
    _check(load().bsg_mma_ceiling(int(iters), _ptr(dstatus), ctypes.byref(flops),
                                  _stream_ptr(stream)), "bsg_mma_ceiling")
    return float(flops.value)


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(load().bsg_launch_count())


def bsgemm_i8_quantize(A, B, workspace, transA: bool = False, transB: bool = False,
                       stream=None, dstatus=None):
    """Step 1 into `workspace` (a Workspace); returns (M, N, K)."""
    torch = _torch()
    _need(A, torch.float32, "A")
    _need(B, torch.float32, "B")
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    K2, N = (B.shape[1], B.shape[0]) if transB else B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    lib = load()
    wp, wn = workspace.ptr_size(lib.bsgemm_i8_workspace_size(M, N, K))
    _check(lib.bsgemm_i8_quantize(_ptr(A), A.shape[1], int(bool(transA)), _ptr(B), B.shape[1],
                                  int(bool(transB)), M, N, K, wp, wn, _ptr(dstatus),
                                  _stream_ptr(stream)), "bsgemm_i8_quantize")
    return M, N, K


def bsgemm_i8_contract(M, N, K, C, workspace, relu: bool = False, stream=None, dstatus=None):
    """Steps 2-3 from `workspace` into the M x N float32 tensor C."""
    lib = load()
    wp, wn = workspace.ptr_size(lib.bsgemm_i8_workspace_size(M, N, K))
    _check(lib.bsgemm_i8_contract(M, N, K, int(bool(relu)), _ptr(C), C.shape[1], wp, wn,
                                  _ptr(dstatus), _stream_ptr(stream)), "bsgemm_i8_contract")
    return C


def bsgemm_i8_host(A, B, relu: bool = False, out=None, stream=None, workspace=None):
    """The unit on HOST float32 tensors (pinned for asynchronous copies);
    returns (C on the host, device status bits).  Synchronizes the stream."""
    torch = _torch()
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or t.is_cuda or t.dim() != 2 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous 2-D float32 host tensor")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    lib = load()
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    wp, wn = _ws(workspace, lib.bsgemm_i8_host_workspace_size(M, N, K))
    st = ctypes.c_int32(0)
    _check(lib.bsgemm_i8_host(_ptr(A), _ptr(B), M, N, K, int(bool(relu)), _ptr(C), wp, wn,
                              ctypes.byref(st), _stream_ptr(stream)), "bsgemm_i8_host")
    return C, st.value


def bsgemm_i8_host_batch(items, stream=None, workspace=None):
    """Several independent units on HOST float32 tensors in one pipelined
    call.  `items`: tuples (A, B, relu) or (A, B, relu, out) of contiguous
    host tensors (pinned for asynchronous copies).  Returns (list of C on the
    host, OR of the device status bits).  Synchronizes the stream."""
    torch = _torch()
    lib = load()
    n = len(items)
    arr = (HostItem * n)()
    dims, offs, outs = [], [], []
    total = 0
    for it in items:
        A, B = it[0], it[1]
        for name, t in (("A", A), ("B", B)):
            if t.dtype != torch.float32 or t.is_cuda or t.dim() != 2 or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous 2-D float32 host tensor")
        M, K = A.shape
        K2, N = B.shape
        if K != K2:
            raise ValueError("inner dimensions differ")
        dims.append((M, N, K))
        offs.append(total)
        total += (lib.bsgemm_i8_host_workspace_size(M, N, K) + 255) // 256 * 256
    # one device workspace carved into the items' parts, kept beyond the call
    wp, wn = _ws(workspace, total)
    base = wp.value
    for i, (it, (M, N, K)) in enumerate(zip(items, dims)):
        C = it[3] if len(it) > 3 and it[3] is not None else torch.empty(
            (M, N), dtype=torch.float32, pin_memory=True)
        outs.append(C)
        arr[i] = HostItem(it[0].data_ptr(), it[1].data_ptr(), M, N, K, int(bool(it[2])),
                          C.data_ptr(), base + offs[i], lib.bsgemm_i8_host_workspace_size(M, N, K))
    st = ctypes.c_int32(0)
    _check(lib.bsgemm_i8_host_batch(arr, n, ctypes.byref(st), _stream_ptr(stream)),
           "bsgemm_i8_host_batch")
    return outs, st.value


def hash_f32(C, stream=None, workspace=None) -> bytes:
    """32-byte tree hash of a float32 matrix's bytes (synchronizes)."""
    torch = _torch()
    _need(C, torch.float32, "C")
    M, N = C.shape
    lib = load()
    out = torch.empty(32, dtype=torch.uint8, device=C.device)
    wp, wn = _ws(workspace, lib.bsg_hash_f32_workspace_size(M, N))
    _check(lib.bsg_hash_f32(_ptr(C), M, N, N, _ptr(out), wp, wn, _stream_ptr(stream)),
           "bsg_hash_f32")
    return bytes(out.cpu().tolist())


def audit(A, B, C, relu=False, seed: int = 0, nsamples: int = 256, mismatches=None,
          cells=None, stream=None):
    """Live audit of C = bsgemm_i8(A, B, relu): `nsamples` seeded cells
    recomputed on the CUDA cores; mismatches are added to the device uint32
    tensor `mismatches` (a fresh zero one if None), which is returned.
    `cells` (int64, 2 * nsamples elements, or None) receives the sampled
    (row, column) pairs."""
    torch = _torch()
    _need(A, torch.float32, "A")
    _need(B, torch.float32, "B")
    _need(C, torch.float32, "C")
    M, K = A.shape
    K2, N = B.shape
    if K != K2 or tuple(C.shape) != (M, N):
        raise ValueError("shapes differ")
    if mismatches is None:
        mismatches = torch.zeros(1, dtype=torch.int32, device=A.device)
    if cells is not None and (cells.dtype != torch.int64 or cells.numel() < 2 * nsamples):
        raise ValueError("cells must be an int64 tensor of 2 * nsamples elements")
    _check(load().bsg_audit(_ptr(A), K, _ptr(B), N, _ptr(C), N, M, N, K, int(bool(relu)),
                            ctypes.c_uint64(seed), int(nsamples), _ptr(mismatches), _ptr(cells),
                            _stream_ptr(stream)), "bsg_audit")
    return mismatches


def bsgemm_i8_group(items, dstatus=None, stream=None, workspace=None):
    """Several units in one GEMM launch.  `items`: up to 3 tuples
    (A, B, transA, transB, relu) of CUDA float32 tensors as for bsgemm_i8_ex
    (A stored M x K, or K x M with transA; B stored K x N, or N x K with
    transB).  Returns the list of C tensors."""
    torch = _torch()
    lib = load()
    n = len(items)
    arr = (GemmItem * n)()
    dims, outs, offs = [], [], []
    total = 0
    for A, B, tA, tB, relu in items:
        _need(A, torch.float32, "A")
        _need(B, torch.float32, "B")
        M, K = (A.shape[1], A.shape[0]) if tA else (A.shape[0], A.shape[1])
        N = B.shape[0] if tB else B.shape[1]
        dims.append((M, N, K))
        offs.append(total)
        total += (lib.bsgemm_i8_workspace_size(M, N, K) + 255) // 256 * 256
    # one workspace carved into the items' parts (the library's default one
    # unless `workspace` is given), kept alive beyond this call
    wp, wn = _ws(workspace, total)
    base = wp.value
    for i, ((A, B, tA, tB, relu), (M, N, K)) in enumerate(zip(items, dims)):
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
        outs.append(C)
        size = lib.bsgemm_i8_workspace_size(M, N, K)
        arr[i] = GemmItem(A.data_ptr(), A.shape[1], int(bool(tA)), B.data_ptr(), B.shape[1],
                          int(bool(tB)), M, N, K, int(bool(relu)), C.data_ptr(), N,
                          base + offs[i], size)
    _check(lib.bsgemm_i8_group(arr, n, _ptr(dstatus), _stream_ptr(stream)), "bsgemm_i8_group")
    return outs


def wquant_cols(W, bits: int = 8, pow2: bool = False, dstatus=None, stream=None,
                workspace=None):
    """Weight storage codes of a K x N f32 weight (per-column scales):
    (Q, scale).  bits 8: Q int8 K x N; bits 4: Q uint8 K x ceil(N/2), two
    4-bit codes per byte."""
    torch = _torch()
    _need(W, torch.float32, "W")
    K, N = W.shape
    if bits == 8:
        Q = torch.empty((K, N), dtype=torch.int8, device=W.device)
    else:
        Q = torch.empty((K, (N + 1) // 2), dtype=torch.uint8, device=W.device)
    sc = torch.empty(N, dtype=torch.float32, device=W.device)
    lib = load()
    wp, wn = _ws(workspace, lib.bsg_wquant_cols_workspace_size(K, N))
    _check(lib.bsg_wquant_cols(_ptr(W), K, N, N, int(bits), int(bool(pow2)), _ptr(Q),
                               Q.shape[1], _ptr(sc), wp, wn, _ptr(dstatus), _stream_ptr(stream)),
           "bsg_wquant_cols")
    return Q, sc


def wdequant_cols(Q, scale, N: int, bits: int = 8, stream=None):
    """The stored weights f32(q * s) (K x N f32)."""
    torch = _torch()
    K = Q.shape[0]
    out = torch.empty((K, N), dtype=torch.float32, device=Q.device)
    _check(load().bsg_wdequant_cols(_ptr(Q), K, N, Q.shape[1], int(bits), _ptr(scale),
                                    _ptr(out), N, _stream_ptr(stream)), "bsg_wdequant_cols")
    return out


def selftest(workspace=None):
    """The init gate: (status, audit mismatches, hash matched).  Synchronous."""
    lib = load()
    wp, wn = _ws(workspace, lib.bsg_selftest_workspace_size())
    mis = ctypes.c_uint32(0)
    ok = ctypes.c_int(0)
    st = lib.bsg_selftest(wp, wn, ctypes.byref(mis), ctypes.byref(ok))
    return int(st), int(mis.value), bool(ok.value)


def probe_hash_async(seed: int, M: int = 1024, N: int = 1024, K: int = 1024, out=None,
                     stream=None, dstatus=None, workspace=None):
    """The probe hash into a 32-byte device tensor (asynchronous)."""
    torch = _torch()
    lib = load()
    out = out if out is not None else torch.empty(32, dtype=torch.uint8, device="cuda")
    wp, wn = _ws(workspace, lib.bsg_probe_workspace_size(M, N, K))
    _check(lib.bsg_probe_hash_async(ctypes.c_uint64(seed), M, N, K, _ptr(out), wp, wn,
                                    _ptr(dstatus), _stream_ptr(stream)), "bsg_probe_hash_async")
    return out


def probe_hash(seed: int, M: int = 1024, N: int = 1024, K: int = 1024, stream=None,
               workspace=None) -> bytes:
    """The probe hash as 32 host bytes (synchronizes)."""
    lib = load()
    buf = (ctypes.c_uint8 * 32)()
    wp, wn = _ws(workspace, lib.bsg_probe_workspace_size(M, N, K))
    _check(lib.bsg_probe_hash(ctypes.c_uint64(seed), M, N, K, buf, wp, wn, _stream_ptr(stream)),
           "bsg_probe_hash")
    return bytes(buf)
