"""The multi-rank host path on the CPU: world-size-2 gloo ranks.

The unit shards by rows without any exchange; the only cross-rank step is
the probe-hash comparison of "Layer 3: the kernel probe".  Here two ranks
each compute the oracle's result for their row shard of one problem and
their probe hash: the shards reassemble the whole, the hashes agree, a
tampered rank is detected, and the max-over-ranks reduction takes the
slowest rank's time.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from verifiable_quantize_rows_gb300.replicas import row_shard


def test_row_shard_covers_exactly():
    for M in (0, 1, 7, 8192, 8193):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                a, b = row_shard(M, r, world)
                assert 0 <= a <= b <= M
                seen.extend(range(a, b))
            assert seen == list(range(M))
    with pytest.raises(ValueError):
        row_shard(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, tamper, out):
    import torch
    import torch.distributed as dist
    import oracle
    from verifiable_quantize_rows_gb300 import inputs
    from verifiable_quantize_rows_gb300.replicas import max_over_ranks, probe_hashes_agree
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    orc = oracle.load()
    A = inputs.gpt2_activations(96, 64, 3, outlier_frac=0.05).numpy()
    B = inputs.gpt2_weights(64, 40, 3).numpy()
    a, b = row_shard(A.shape[0], rank, world)
    C, st = orc.bsgemm_i8(A[a:b], B)
    pieces = [None] * world
    dist.all_gather_object(pieces, (a, C.tobytes()))
    h, _ = orc.probe_hash(5, 33, 17, 70)
    if tamper and rank == 1:
        h = bytes([h[0] ^ 1]) + h[1:]
    agree, hexes = probe_hashes_agree(h)
    t = max_over_ranks([1.0 + rank, 5.0 - rank])
    if rank == 0:
        full, _ = orc.bsgemm_i8(A, B)
        pieces.sort()
        got = np.concatenate([np.frombuffer(p, np.float32).reshape(-1, B.shape[1]) for _, p in pieces])
        out.put((bool(np.array_equal(got.view(np.uint32), full.view(np.uint32))), agree, t))
    dist.destroy_process_group()


@pytest.mark.parametrize("tamper", [False, True])
def test_two_gloo_ranks(tamper):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, tamper, q)) for r in range(2)]
    for p in procs:
        p.start()
    shards_ok, agree, t = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert shards_ok
    assert agree == (not tamper)
    assert t == [2.0, 5.0]
