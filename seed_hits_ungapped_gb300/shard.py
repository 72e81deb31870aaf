"""Seed-range sharding of one query batch across ranks (one GPU per rank).

Query seeds are independent, so a batch splits into contiguous seed ranges.
Rank r takes seeds [s0, s1) and the query bases [s0, s1 + span - 1) they
read; its anchors carry query coordinates local to that slice (add s0) and its
anchor ids are local (add the exclusive scan of the lower ranks' totals).  The
only exchange is that scan of per-rank 64-bit totals, which also applies the
32-bit hit-index refusal to the whole batch.  No collective touches the data
path.
"""
from __future__ import annotations

MAX_HIT_INDEX = (1 << 32) - 1


def seed_range(query_len: int, span: int, world: int, rank: int):
    """(s0, s1, q0, q1): this rank's seeds [s0, s1) and query slice [q0, q1)."""
    n_seeds = max(0, query_len - span + 1)
    s0 = n_seeds * rank // world
    s1 = n_seeds * (rank + 1) // world
    if s1 <= s0:
        return s0, s0, s0, s0
    return s0, s1, s0, s1 + span - 1


def global_offsets(local_total: int, group=None):
    """(id_base, global_total) from an all-gather of the per-rank totals.

    Raises OverflowError when the batch as a whole does not fit the 32-bit
    hit index (the refusal of "C. Hit discovery", C.2, applied globally).
    """
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        totals = [int(local_total)]
        rank = 0
    else:
        t = torch.tensor([int(local_total)], dtype=torch.int64)
        world = dist.get_world_size(group)
        bufs = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(bufs, t, group=group)
        totals = [int(b.item()) for b in bufs]
        rank = dist.get_rank(group)
    base = sum(totals[:rank])
    total = sum(totals)
    if total > MAX_HIT_INDEX:
        raise OverflowError("batch total %d exceeds the 32-bit hit index" % total)
    return base, total
