"""CPU oracle for the block-scaled int8 GEMM -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``bsg_oracle.c`` (plain C99, compiled with
``-ffp-contract=off -fno-fast-math``); this module builds it with gcc and
wraps it with ctypes over numpy arrays.  Only the test suite, the smoke check
and the benchmark's CPU-baseline leg may import this package.  It shares no
code with the CUDA library and never imports it.

What each function computes, and the page passage it follows, is stated in
``bsg_oracle.c``.  Pins (the checks that tie this oracle to something other
than itself) live in ``tests/``.  Parity status per function:

* quantize (scale, inv, int8 values): pinned by the exact-rational IEEE-754
  referee and by constructed ties; the inv derivation (reading R2) is a
  reading of a silent passage, so its agreement with the pages' own system is
  unpinned -- the tests pin only that the reading is what is computed.
* integer contraction: pinned by big-integer brute force and the unit-scale
  absolute.
* epilogue and ReLU: pinned by the exact-rational referee.
* BLAKE2s / tree hash: pinned by the RFC 7693 test vector and Python's
  hashlib.blake2s (which implements the tree parameters).
* SplitMix64 probe inputs: pinned by the generator's published outputs.
* probe hash as a whole: "parity unpinned" against the pages' system (the
  pages give neither the probe's inputs nor its hash function).
* presk weight storage (scales, int8 / int4 codes, stored weights): pinned by
  exact rationals (the scale's f32 rounding, the nearest integer with ties to
  even, subnormal channels included), constructed ties, the page's error
  rule, pow2 exactness and the nibble layout.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsg_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libbsg_oracle.so")

CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-fopenmp"]

ORC_OK = 0
ORC_ERR_ARG = 1
ORC_ERR_RANGE = 2
ORC_ERR_NONFINITE = 5

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str, out: str, extra: list[str] | None = None) -> str:
    """Compile an oracle source file into a shared library (gcc)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, *(extra or []), src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or (
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            tmp = _LIB_PATH + f".{os.getpid()}.tmp"
            compile_oracle(_SRC, tmp)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_I8P = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_I32P = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_I64P = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_U8P = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def _declare(lib):
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_scale_from_max.argtypes = [ctypes.c_float, ctypes.POINTER(ctypes.c_float),
                                       ctypes.POINTER(ctypes.c_float)]
    lib.orc_scales_from_max.argtypes = [_F32P, _i64, _F32P, _F32P]
    lib.orc_quantize_value.argtypes = [ctypes.c_float, ctypes.c_float]
    lib.orc_quantize_value.restype = ctypes.c_int
    lib.orc_quantize_rows.argtypes = [_F32P, _i64, _i64, _i64, _I8P, _i64, _F32P, _F32P]
    lib.orc_quantize_cols.argtypes = [_F32P, _i64, _i64, _i64, _I8P, _i64, _F32P, _F32P]
    lib.orc_gemm_s32.argtypes = [_I8P, _I8P, _i64, _i64, _i64, _I32P]
    lib.orc_epi.argtypes = [ctypes.c_int32, ctypes.c_float, ctypes.c_float]
    lib.orc_epi.restype = ctypes.c_float
    lib.orc_relu.argtypes = [ctypes.c_float]
    lib.orc_relu.restype = ctypes.c_float
    lib.orc_epilogue.argtypes = [_I32P, _F32P, _F32P, _i64, _i64, ctypes.c_int, _F32P]
    lib.orc_bsgemm_i8.argtypes = [_F32P, _F32P, _i64, _i64, _i64, ctypes.c_int, _F32P,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.orc_bsgemm_cells.argtypes = [_F32P, _F32P, _i64, _i64, _i64, ctypes.c_int, _I64P,
                                     _I64P, _i64, _F32P, ctypes.c_void_p]
    lib.orc_blake2s.argtypes = [ctypes.c_char_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, _U8P]
    lib.orc_tree_hash.argtypes = [ctypes.c_char_p, ctypes.c_size_t, _U8P]
    lib.orc_hash_f32.argtypes = [_F32P, _i64, _i64, _i64, _U8P]
    lib.orc_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    lib.orc_splitmix64.restype = ctypes.c_uint64
    lib.orc_probe_value.argtypes = [ctypes.c_uint64]
    lib.orc_probe_value.restype = ctypes.c_float
    lib.orc_probe_inputs.argtypes = [ctypes.c_uint64, _i64, _i64, _i64, _F32P, _F32P]
    lib.orc_probe_hash.argtypes = [ctypes.c_uint64, _i64, _i64, _i64, _U8P]
    lib.orc_pow2_ceil.argtypes = [ctypes.c_float]
    lib.orc_pow2_ceil.restype = ctypes.c_float
    lib.orc_wquant_cols.argtypes = [_F32P, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _I8P,
                                    _i64, _F32P]
    lib.orc_wquant_cols.restype = ctypes.c_int
    lib.orc_pack_int4.argtypes = [_I8P, _i64, _i64, _i64, _U8P, _i64]
    lib.orc_wdequant_cols.argtypes = [_I8P, _i64, _i64, _i64, _F32P, _F32P, _i64]
    for name in ("orc_quantize_rows", "orc_quantize_cols", "orc_gemm_s32", "orc_epilogue",
                 "orc_bsgemm_i8", "orc_bsgemm_cells", "orc_hash_f32", "orc_probe_hash"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first if needed).

    ``path`` selects another build of the oracle source (the mutation tests
    load deliberately broken copies this way); the default build is cached.
    """
    global _lib
    if path is not None:
        return Oracle(_declare(ctypes.CDLL(path)))
    if _lib is None:
        _lib = Oracle(_declare(ctypes.CDLL(build())))
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """numpy front end of one loaded oracle library."""

    def __init__(self, lib):
        self.lib = lib

    def num_threads(self) -> int:
        return int(self.lib.orc_num_threads())

    # -- step 1: scales and the quantize rule ----------------------------
    def scale_from_max(self, m: float) -> tuple[float, float]:
        s, i = ctypes.c_float(), ctypes.c_float()
        self.lib.orc_scale_from_max(ctypes.c_float(m), ctypes.byref(s), ctypes.byref(i))
        return s.value, i.value

    def scales_from_max(self, m):
        m = _c(m, np.float32).reshape(-1)
        sc = np.zeros(max(len(m), 1), np.float32)
        iv = np.zeros(max(len(m), 1), np.float32)
        self.lib.orc_scales_from_max(m if len(m) else np.zeros(1, np.float32), len(m), sc, iv)
        return sc[:len(m)], iv[:len(m)]

    def quantize_value(self, x: float, inv: float) -> int:
        return int(self.lib.orc_quantize_value(ctypes.c_float(x), ctypes.c_float(inv)))

    def quantize_rows(self, A):
        A = _c(A, np.float32)
        M, K = A.shape
        Q = np.zeros((M, K), np.int8)
        sc = np.zeros(max(M, 1), np.float32)
        iv = np.zeros(max(M, 1), np.float32)
        st = self.lib.orc_quantize_rows(A, M, K, K, Q, K, sc, iv)
        return Q, sc[:M], iv[:M], st

    def quantize_cols(self, B):
        B = _c(B, np.float32)
        K, N = B.shape
        Q = np.zeros((K, N), np.int8)
        sc = np.zeros(max(N, 1), np.float32)
        iv = np.zeros(max(N, 1), np.float32)
        st = self.lib.orc_quantize_cols(B, K, N, N, Q, N, sc, iv)
        return Q, sc[:N], iv[:N], st

    # -- step 2: the exact integer contraction ---------------------------
    def gemm_s32(self, Aq, Bq):
        Aq, Bq = _c(Aq, np.int8), _c(Bq, np.int8)
        M, K = Aq.shape
        K2, N = Bq.shape
        assert K == K2
        S = np.zeros((M, N), np.int32)
        st = self.lib.orc_gemm_s32(Aq, Bq, M, N, K, S)
        return S, st

    # -- step 3: the epilogue --------------------------------------------
    def epi(self, s: int, a: float, b: float) -> float:
        return float(self.lib.orc_epi(int(s), ctypes.c_float(a), ctypes.c_float(b)))

    def relu(self, c: float) -> float:
        return float(self.lib.orc_relu(ctypes.c_float(c)))

    def epilogue(self, S, sa, sb, relu: bool):
        S = _c(S, np.int32)
        M, N = S.shape
        C = np.zeros((M, N), np.float32)
        self.lib.orc_epilogue(S, _c(sa, np.float32).reshape(-1) if M else np.zeros(1, np.float32),
                              _c(sb, np.float32).reshape(-1) if N else np.zeros(1, np.float32),
                              M, N, int(bool(relu)), C)
        return C

    # -- the whole unit ---------------------------------------------------
    def bsgemm_i8(self, A, B, relu: bool = False, want_s: bool = False):
        A, B = _c(A, np.float32), _c(B, np.float32)
        M, K = A.shape
        K2, N = B.shape
        assert K == K2
        C = np.zeros((M, N), np.float32)
        S = np.zeros((M, N), np.int32) if want_s else None
        st = self.lib.orc_bsgemm_i8(A, B, M, N, K, int(bool(relu)), C,
                                    S.ctypes.data if want_s else None, None, None)
        return (C, S, st) if want_s else (C, st)

    def bsgemm_cells(self, A, B, rows, cols, relu: bool = False):
        A, B = _c(A, np.float32), _c(B, np.float32)
        M, K = A.shape
        _, N = B.shape
        rows, cols = _c(rows, np.int64), _c(cols, np.int64)
        out = np.zeros(max(len(rows), 1), np.float32)
        S = np.zeros(max(len(rows), 1), np.int32)
        st = self.lib.orc_bsgemm_cells(A, B, M, N, K, int(bool(relu)), rows, cols, len(rows),
                                       out, S.ctypes.data)
        return out[:len(rows)], S[:len(rows)], st

    # -- the probe ---------------------------------------------------------
    def blake2s(self, data: bytes, fanout=1, depth=1, leaf_size=0, node_offset=0,
                node_depth=0, inner_size=0, last_node=False) -> bytes:
        out = np.zeros(32, np.uint8)
        self.lib.orc_blake2s(data, len(data), fanout, depth, leaf_size, node_offset, node_depth,
                             inner_size, int(bool(last_node)), out)
        return out.tobytes()

    def tree_hash(self, data: bytes) -> bytes:
        out = np.zeros(32, np.uint8)
        self.lib.orc_tree_hash(data, len(data), out)
        return out.tobytes()

    def hash_f32(self, C) -> bytes:
        C = _c(C, np.float32)
        M, N = C.shape
        out = np.zeros(32, np.uint8)
        self.lib.orc_hash_f32(C if C.size else np.zeros(1, np.float32), M, N, N, out)
        return out.tobytes()

    def splitmix64(self, seed: int, i: int) -> int:
        return int(self.lib.orc_splitmix64(seed, i))

    def probe_value(self, z: int) -> float:
        return float(self.lib.orc_probe_value(z))

    def probe_inputs(self, seed: int, M: int, N: int, K: int):
        A = np.zeros((M, K), np.float32)
        B = np.zeros((K, N), np.float32)
        self.lib.orc_probe_inputs(seed, M, N, K, A, B)
        return A, B

    def probe_hash(self, seed: int, M: int, N: int, K: int) -> tuple[bytes, int]:
        out = np.zeros(32, np.uint8)
        st = self.lib.orc_probe_hash(seed, M, N, K, out)
        return out.tobytes(), st

    # -- presk weight storage ("Precision" manual, "Integer weights") ------
    def pow2_ceil(self, s: float) -> float:
        return float(self.lib.orc_pow2_ceil(s))

    def wquant_cols(self, W, bits: int = 8, pow2: bool = False):
        """Codes (K x N int8), per-column scales and status."""
        W = _c(W, np.float32)
        K, N = W.shape
        Q = np.zeros((K, N), np.int8)
        sc = np.zeros(N, np.float32)
        st = self.lib.orc_wquant_cols(W, K, N, N, int(bits), int(bool(pow2)), Q, N, sc)
        return Q, sc, st

    def pack_int4(self, Q):
        Q = _c(Q, np.int8)
        K, N = Q.shape
        P = np.zeros((K, (N + 1) // 2), np.uint8)
        self.lib.orc_pack_int4(Q, K, N, N, P, (N + 1) // 2)
        return P

    def wdequant_cols(self, Q, scale):
        Q = _c(Q, np.int8)
        K, N = Q.shape
        out = np.zeros((K, N), np.float32)
        self.lib.orc_wdequant_cols(Q, K, N, N, _c(scale, np.float32), out, N)
        return out
