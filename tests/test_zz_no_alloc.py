"""bsgemm_i8_noalloc: the unit for callers that cannot allocate device
memory -- a framework that owns every device allocation and lends none to
extensions, or an embedding where the library may not touch the allocator.
Its scratch is a device array compiled into the library, so it takes no
workspace.

Checked through the C ABI, on calls in a row with different inputs: its
output is bit-identical to the CPU oracle's and to bsgemm_i8's on a
caller-provided workspace (the tolerance of every parity test here:
bitwise).  The calls cover the fused quantize launch (K = 768), the separate
row and column quantizes (K = 3072) and the two-pass column quantize whose
partial maxima live in the shared array (K > 4096).  Problems too large for
the array are rejected before anything runs.  This file is collected last so
a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal
import verifiable_quantize_rows_gb300 as bsg
from verifiable_quantize_rows_gb300 import inputs

pytestmark = pytest.mark.gpu


def _entry():
    fn = bsg.load().bsgemm_i8_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _noalloc(fn, A, B, relu):
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(A.data_ptr(), B.data_ptr(), M, N, K, int(relu), C.data_ptr(), st.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, bsg.STATUS.get(rc, rc)
    torch.cuda.synchronize()
    return C, int(st.item())


CALLS = [
    ("fc", 8192, 3072, 768, True, 2),
    ("proj", 8192, 768, 3072, False, 3),
    ("long columns", 256, 320, 5000, False, 21),
]


def test_noalloc_matches_oracle_and_workspace_entry_point_on_calls_in_a_row(orc):
    fn = _entry()
    for name, M, N, K, relu, seed in CALLS:
        A = inputs.gpt2_activations(M, K, seed)
        B = inputs.gpt2_weights(K, N, seed)
        Ad, Bd = A.cuda(), B.cuda()
        got, st = _noalloc(fn, Ad, Bd, relu)
        assert st == 0
        want = bsg.bsgemm_i8(Ad, Bd, relu=relu)
        torch.cuda.synchronize()
        Co, _ = orc.bsgemm_i8(A.numpy(), B.numpy(), relu)
        g = got.cpu().numpy()
        assert_bits_equal(g, Co, f"{name}: noalloc vs oracle")
        assert_bits_equal(g, want.cpu().numpy(), f"{name}: noalloc vs bsgemm_i8")


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _entry()
    lib = bsg.load()
    M, N, K = 8192, 50304, 768          # the LM head needs ~90 MB of scratch
    assert lib.bsgemm_i8_workspace_size(M, N, K) > (64 << 20)
    x = torch.zeros(1, device="cuda")
    rc = fn(x.data_ptr(), x.data_ptr(), M, N, K, 0, x.data_ptr(), None, None)
    assert rc == 3   # BSG_ERR_WORKSPACE, before anything is launched
