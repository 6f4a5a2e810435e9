"""Host-side logic for running the unit on several GPUs (one process each).

The unit shards without any exchange: rows of A (per-row scales) split
across ranks give disjoint row blocks of C, with B replicated.  The one
cross-rank step is the pages' own: every replica publishes its probe hash
("Verification -- why you can trust the numbers", section "Layer 3: the kernel
probe"), and honest replicas agree.  These helpers take a torch.distributed
process group; they carry no data of the computation itself.
"""
from __future__ import annotations


def row_shard(M: int, rank: int, world: int) -> tuple[int, int]:
    """Rows [start, stop) of an M-row problem owned by `rank` of `world`:
    contiguous, as equal as possible, covering every row exactly once."""
    if world < 1 or not 0 <= rank < world or M < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(M, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(values, group=None, device=None):
    """Element-wise maximum of a list of floats over all ranks (step times)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return [float(x) for x in t.tolist()]


def probe_hashes_agree(digest: bytes, group=None, device=None) -> tuple[bool, list[str]]:
    """Gather every rank's 32-byte probe hash; (all equal, hex digests)."""
    import torch
    import torch.distributed as dist
    if len(digest) != 32:
        raise ValueError("a probe hash is 32 bytes")
    mine = torch.tensor(list(digest), dtype=torch.int32, device=device)
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return True, [digest.hex()]
    allh = [torch.empty_like(mine) for _ in range(dist.get_world_size(group))]
    dist.all_gather(allh, mine, group=group)
    hexes = [bytes(int(v) for v in h.tolist()).hex() for h in allh]
    return all(h == hexes[0] for h in hexes), hexes
