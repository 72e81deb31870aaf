"""Seed-range sharding across ranks (world size 2, gloo on CPU).  Each rank
runs the oracle on its slice; per-rank anchors, with their query coordinates
shifted by the slice start and their ids offset by the exclusive scan of the
lower ranks' totals, must reassemble the single-process result exactly."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
from seed_hits_ungapped_gb300 import shard, synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, outdir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.make("tiny", scale=0.1)
        _, span = oracle.pattern_info()
        s0, s1, q0, q1 = shard.seed_range(w.query.size, span, world, rank)
        res = oracle.run_path(w.ref, w.query[q0:q1], w.matrix, w.xdrop, w.K)
        base, total = shard.global_offsets(int(res["total"]))
        anchors = np.concatenate([c["anchors"] for c in res["per_chunk"]]) if res["per_chunk"] else np.zeros((0, 2), np.uint32)
        ids = np.concatenate([c["ids"] for c in res["per_chunk"]]) if res["per_chunk"] else np.zeros(0, np.uint32)
        anchors = anchors.astype(np.int64)
        anchors[:, 1] += q0
        np.savez(os.path.join(outdir, "r%d.npz" % rank), anchors=anchors, ids=ids.astype(np.int64) + base,
                 base=base, total=total, local=res["total"])
        # the global refusal: a pretend shard total that overflows the hit index
        try:
            shard.global_offsets((1 << 32) - 1 if rank == 1 else 1)
            refused = False
        except OverflowError:
            refused = True
        assert refused
    finally:
        dist.destroy_process_group()


def test_two_rank_seed_shards_reassemble(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    parts = [np.load(os.path.join(tmp_path, "r%d.npz" % r)) for r in range(world)]
    w = synth.make("tiny", scale=0.1)
    whole = oracle.run_path(w.ref, w.query, w.matrix, w.xdrop, w.K)
    want_anchors = np.concatenate([c["anchors"] for c in whole["per_chunk"]]).astype(np.int64)
    want_ids = np.concatenate([c["ids"] for c in whole["per_chunk"]]).astype(np.int64)
    assert parts[0]["base"] == 0 and parts[1]["base"] == parts[0]["local"]
    assert parts[0]["total"] == parts[1]["total"] == whole["total"]
    assert np.array_equal(np.concatenate([p["anchors"] for p in parts]), want_anchors)
    assert np.array_equal(np.concatenate([p["ids"] for p in parts]), want_ids)


def test_seed_range_covers_every_seed_once():
    for L in (0, 5, 19, 20, 1000, 12345):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                s0, s1, q0, q1 = shard.seed_range(L, 19, world, r)
                seen.extend(range(s0, s1))
                if s1 > s0:
                    assert q0 == s0 and q1 == s1 + 18 and q1 <= L
            assert seen == list(range(max(0, L - 18)))
