"""Streams, graphs and host threads.

- Capture into a CUDA graph: bsgemm_i8 on the fused quantize path (K <= 2048),
  on the path that quantizes B on the library's second stream (K > 2048), and
  with B's columns on the one-read item list (K > 4096, its scratch cleared by
  a captured memset),
  and bsgemm_i8_chain (its second weight matrix on that stream too), each
  captured after a first eager call on the device, then replayed with new
  inputs copied into the captured buffers: every replay is bitwise the
  oracle's result for those inputs.
- Host threads: several threads call bsgemm_i8 at once, each on its own
  stream and workspace, on different shapes; every result is bitwise what a
  single-threaded call gives.  (The library serialises its own shared state
  -- the second stream's fork and join, the host-buffer copy streams -- with
  locks; the kernels of different calls share nothing.)
"""
import threading

import numpy as np
import pytest
import torch

from gpu_util import assert_bits_equal, host
from verifiable_quantize_rows_gb300 import inputs
import verifiable_quantize_rows_gb300 as bsg

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(640, 520, 700), (300, 260, 3000), (256, 300, 5000)],
                         ids=lambda v: str(v))
def test_unit_replays_from_a_cuda_graph(orc, M, N, K):
    A = torch.empty(M, K, device="cuda")
    B = torch.empty(K, N, device="cuda")
    C = torch.empty(M, N, device="cuda")
    ws = bsg.Workspace()
    A.copy_(inputs.normal((M, K), 1.0, 1))
    B.copy_(inputs.normal((K, N), 0.1, 2))
    bsg.bsgemm_i8(A, B, relu=True, out=C, workspace=ws)        # first call: eager
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bsg.bsgemm_i8(A, B, relu=True, out=C, workspace=ws)
    for rep in range(2):
        a = inputs.normal((M, K), 1.0, 10 + rep)
        b = inputs.adversarial(N, K, 20 + rep, along_rows=False)
        A.copy_(a)
        B.copy_(b)
        g.replay()
        torch.cuda.synchronize()
        Co, _ = orc.bsgemm_i8(a.numpy(), b.numpy(), True)
        assert_bits_equal(host(C), Co, f"replay {rep}")


def test_chain_replays_from_a_cuda_graph(orc):
    M, K, N1, N2 = 256, 300, 700, 130
    A = torch.empty(M, K, device="cuda")
    B1 = torch.empty(K, N1, device="cuda")
    B2 = torch.empty(N1, N2, device="cuda")
    C1 = torch.empty(M, N1, device="cuda")
    C2 = torch.empty(M, N2, device="cuda")
    ws = bsg.Workspace()
    B1.copy_(inputs.normal((K, N1), 0.1, 3))
    B2.copy_(inputs.normal((N1, N2), 0.1, 4))
    A.copy_(inputs.normal((M, K), 1.0, 5))
    bsg.bsgemm_i8_chain(A, B1, B2, True, False, out1=C1, out2=C2, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bsg.bsgemm_i8_chain(A, B1, B2, True, False, out1=C1, out2=C2, workspace=ws)
    for rep in range(2):
        a = inputs.normal((M, K), 1.0, 30 + rep)
        b2 = inputs.normal((N1, N2), 0.1, 40 + rep)
        A.copy_(a)
        B2.copy_(b2)
        g.replay()
        torch.cuda.synchronize()
        C1o, _ = orc.bsgemm_i8(a.numpy(), host(B1), True)
        C2o, _ = orc.bsgemm_i8(C1o, b2.numpy(), False)
        assert_bits_equal(host(C1), C1o, f"replay {rep} C1")
        assert_bits_equal(host(C2), C2o, f"replay {rep} C2")


def test_concurrent_host_threads():
    shapes = [(512, 384, 700), (300, 520, 2500), (256, 256, 5000), (1000, 96, 64)]
    cases = []
    for i, (M, N, K) in enumerate(shapes):
        A = inputs.normal((M, K), 1.0, 70 + i).cuda()
        B = inputs.adversarial(N, K, 80 + i, along_rows=False).cuda()
        want = bsg.bsgemm_i8(A, B, relu=bool(i % 2))
        cases.append((A, B, bool(i % 2), want))
    torch.cuda.synchronize()
    errors = []

    def worker(idx):
        try:
            A, B, relu, want = cases[idx]
            stream = torch.cuda.Stream()
            ws = bsg.Workspace()
            with torch.cuda.stream(stream):
                for _ in range(4):
                    C = bsg.bsgemm_i8(A, B, relu=relu, workspace=ws, stream=stream)
                stream.synchronize()
            if not torch.equal(C.view(torch.int32), want.view(torch.int32)):
                errors.append(f"thread {idx}: result differs")
        except Exception as e:  # reported below, on the main thread
            errors.append(f"thread {idx}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
