"""Duplicate removal over accepted HSPs on the GPU (hspz_dedup,
hspz_gather_records) against the oracle's dedup.

Integer work: kept indices and final records are compared exactly.  The
criterion itself (equal in all four fields, first in raw order kept) is a
reading of the pages, which give only the funnel counts.
"""
import numpy as np
import pytest

import oracle
from seed_hits_ungapped_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from seed_hits_ungapped_gb300 import hspz
    hspz.load_library()
    return torch


def _dedup_gpu(torch, rec):
    from seed_hits_ungapped_gb300 import hspz
    d = torch.from_numpy(np.ascontiguousarray(rec, np.int32).reshape(-1, 4)).cuda()
    ids = torch.empty(max(1, rec.shape[0]), dtype=torch.int32, device="cuda")
    k = hspz.hspz_dedup(d, rec.shape[0], ids)
    return ids[:k].cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("n,hi,seed", [(1, 3, 0), (1000, 2, 1), (100_000, 3, 2), (300_000, 40, 3), (2_000_000, 6, 4)])
def test_dedup_matches_oracle(torch_cuda, n, hi, seed):
    rng = np.random.default_rng(seed)
    rec = rng.integers(-hi, hi, (n, 4)).astype(np.int32)
    rec[rng.random(n) < 0.01] = [np.iinfo(np.int32).min, -1, np.iinfo(np.int32).max, 0]
    got = _dedup_gpu(torch_cuda, rec)
    assert np.array_equal(got, np.flatnonzero(oracle.dedup(rec)).astype(np.uint32))


def test_dedup_edges_and_capacity(torch_cuda):
    from seed_hits_ungapped_gb300 import hspz
    assert _dedup_gpu(torch_cuda, np.ones((5000, 4), np.int32)).tolist() == [0]
    distinct = np.arange(4 * 7777, dtype=np.int32).reshape(-1, 4)
    assert np.array_equal(_dedup_gpu(torch_cuda, distinct), np.arange(7777, dtype=np.uint32))
    # empty input
    d = torch_cuda.zeros((1, 4), dtype=torch_cuda.int32, device="cuda")
    ids = torch_cuda.zeros(1, dtype=torch_cuda.int32, device="cuda")
    assert hspz.hspz_dedup(d, 0, ids) == 0
    # too small an id buffer: capacity status with the needed count
    rec = np.arange(400, dtype=np.int32).reshape(-1, 4)
    d = torch_cuda.from_numpy(rec).cuda()
    small = torch_cuda.zeros(10, dtype=torch_cuda.int32, device="cuda")
    with pytest.raises(hspz.HspzError) as e:
        hspz.hspz_dedup(d, 100, small)
    assert e.value.status == hspz.HSPZ_E_CAPACITY and e.value.needed == 100


def test_gather_records(torch_cuda):
    from seed_hits_ungapped_gb300 import hspz
    rng = np.random.default_rng(8)
    rec = rng.integers(-1000, 1000, (50_000, 4)).astype(np.int32)
    idx = rng.integers(0, rec.shape[0], 70_001).astype(np.int32)
    out = torch_cuda.empty((idx.size, 4), dtype=torch_cuda.int32, device="cuda")
    hspz.hspz_gather_records(torch_cuda.from_numpy(rec).cuda(), torch_cuda.from_numpy(idx).cuda(), idx.size, out)
    assert np.array_equal(out.cpu().numpy(), rec[idx])


def _run(torch, w, qry, xdrop=None, K=None, max_hits=0):
    from seed_hits_ungapped_gb300.engine import HspEngine
    xdrop = w.xdrop if xdrop is None else xdrop
    K = w.K if K is None else K
    eng = HspEngine(w.ref, w.matrix, xdrop, K)
    gpu = eng.run(torch.from_numpy(qry).cuda(), max_hits=max_hits, keep=True, dedup=True)
    orc = oracle.run_path(w.ref, qry, w.matrix, xdrop, K, max_hits=max_hits)
    return gpu, orc


@pytest.mark.parametrize("name,scale", [("tiny", 1.0), ("mid", 0.05), ("dense", 0.03), ("chunking", 0.02)])
def test_path_final_hsps_match_oracle(torch_cuda, name, scale):
    w = synth.make(name, scale=scale)
    for qry in w.queries:
        gpu, orc = _run(torch_cuda, w, qry, max_hits=w.max_hits)
        assert gpu.n_accepted == orc["accepted_rec"].shape[0]
        assert gpu.n_final == orc["final_rec"].shape[0] <= gpu.n_accepted
        assert gpu.n_final < gpu.n_accepted or gpu.n_accepted == 0
        assert np.array_equal(gpu.final_idx, orc["final_idx"])
        assert np.array_equal(gpu.final_records, orc["final_rec"])


def test_exact_copy_gives_one_final_hsp(torch_cuda):
    rng = np.random.default_rng(21)
    ref = rng.integers(0, 4, 20_000).astype(np.uint8)
    qry = np.concatenate([np.full(50, 4, np.uint8), ref[7_000:7_300], np.full(50, 4, np.uint8)])
    w = synth.Workload(name="copy", ref=ref, queries=[qry], matrix=synth.hoxd70(), xdrop=910, K=3000)
    gpu, orc = _run(torch_cuda, w, qry)
    assert gpu.n_accepted > 100
    assert gpu.final_records.tolist() == orc["final_rec"].tolist()
    assert gpu.final_records.shape[0] == 1 and gpu.final_records[0, :3].tolist() == [7_000, 50, 299]
