"""bsgemm_i8_noalloc: the unit for callers that cannot allocate device
memory (a framework that owns every allocation and lends none, code running
while a stream is captured into a CUDA graph, an embedding that may not touch
the allocator).  Its scratch is a device array compiled into the library, so
it takes no workspace.

Checked through the C ABI: on two calls in a row, with different inputs, its
output is bit-identical to bsgemm_i8's on a caller-provided workspace (the
tolerance of every parity test here: bitwise); problems too large for the
array are rejected before anything runs.  This file is collected last so a
run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    fn = _entry()
    calls = [("fc", 8192, 3072, 768, True, 2), ("proj", 8192, 768, 3072, False, 3)]
    for name, M, N, K, relu, seed in calls:
        A = inputs.gpt2_activations(M, K, seed).cuda()
        B = inputs.gpt2_weights(K, N, seed).cuda()
        want = bsg.bsgemm_i8(A, B, relu=relu)
        torch.cuda.synchronize()
        got, st = _noalloc(fn, A, B, relu)
        assert st == 0
        g = got.cpu().numpy().view(np.uint32)
        w = want.cpu().numpy().view(np.uint32)
        assert np.array_equal(g, w), f"{name}: {(g != w).sum()} cells differ"


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _entry()
    lib = bsg.load()
    M, N, K = 8192, 50304, 768          # the LM head needs ~90 MB of scratch
    assert lib.bsgemm_i8_workspace_size(M, N, K) > (64 << 20)
    x = torch.zeros(1, device="cuda")
    rc = fn(x.data_ptr(), x.data_ptr(), M, N, K, 0, x.data_ptr(), None, None)
    assert rc == 3   # BSG_ERR_WORKSPACE, before anything is launched
