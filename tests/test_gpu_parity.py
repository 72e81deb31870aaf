"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Integer work throughout, so every comparison is bit-exact: prefix, chunk list,
anchors, flags, survivor ids, SegmentPairs, done flags and accepted ids.
Oracle-sized cases are compared element by element; the full-size workload in
the benchmark's launch configuration is compared on the full prefix and on
sampled anchors, flags and records computed one by one by the oracle.
"""
import os

import numpy as np
import pytest

import oracle
from seed_hits_ungapped_gb300 import synth

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from seed_hits_ungapped_gb300 import hspz
    hspz.load_library()  # fails loudly when the library is missing
    return torch


def _engine(torch_cuda, ref, matrix, xdrop, K, pattern=oracle.SEED_PATTERN):
    from seed_hits_ungapped_gb300.engine import HspEngine
    return HspEngine(ref, matrix, xdrop, K, pattern=pattern)


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def assert_same_as_oracle(gpu, orc):
    assert orc["rc"] == 0
    assert gpu.total_hits == orc["total"]
    assert np.array_equal(gpu.prefix, orc["P"])
    assert np.array_equal(gpu.chunks, orc["chunks"])
    assert len(gpu.per_chunk) == len(orc["per_chunk"])
    for g, o in zip(gpu.per_chunk, orc["per_chunk"]):
        assert np.array_equal(g.anchors, o["anchors"])
        assert np.array_equal(g.flags, o["flags"])
        assert np.array_equal(g.ids, o["ids"])
        assert np.array_equal(g.records, o["rec"])
        assert np.array_equal(g.done, o["done"])
        assert np.array_equal(g.accepted, o["accepted"])


def run_both(torch, ref, qry, matrix, xdrop, K, max_hits=0, pattern=oracle.SEED_PATTERN, walk_full=False):
    eng = _engine(torch, ref, matrix, xdrop, K, pattern)
    gpu = eng.run(_dev(torch, qry), max_hits=max_hits, walk_full=walk_full, keep=True)
    orc = oracle.run_path(ref, qry, matrix, xdrop, K, max_hits=max_hits, pattern=pattern)
    return gpu, orc


# ------------------------------------------------------------------ worked example

def test_worked_example_on_gpu(torch_cuda):
    """Counts 0 3 1 0 5 from the figure of "C. Hit discovery": a one-base seed
    over reference CCCGTTTTT and query ACGNT puts 0, 3, 1, 0 and 5 reference
    occurrences behind seeds 0..4."""
    from seed_hits_ungapped_gb300 import hspz
    rows, slots = {}, {}
    for line in open(os.path.join(HERE, "golden", "hit_discovery_worked_example.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, *v = line.split()
            v = [int(x) for x in v]
            if k == "slots":
                slots[v[0]] = v[1:]
            else:
                rows[k] = v
    ref = np.array([1, 1, 1, 2, 3, 3, 3, 3, 3], np.uint8)
    qry = np.array([0, 1, 2, 4, 3], np.uint8)
    torch = torch_cuda
    index = hspz.hspz_build_index(_dev(torch, ref), "1")
    plan = hspz.hspz_find_hits(index, _dev(torch, qry))
    P = plan.prefix().cpu().numpy().view(np.uint32)
    assert P.tolist() == rows["prefix"]
    assert plan.total_hits == 9 and plan.chunks.tolist() == [[0, 5, 0, 9]]
    for mode in (hspz.HSPZ_EXPAND_SPARSE, hspz.HSPZ_EXPAND_DENSE, hspz.HSPZ_EXPAND_AUTO):
        a = torch.full((9, 2), -1, dtype=torch.int32, device="cuda")
        hspz.hspz_expand(plan, 0, a, mode)
        a = a.cpu().numpy()
        bucket_start = {1: 0, 2: 3, 4: 4}  # reference position of occurrence j = 0
        for s, want in slots.items():
            for j, slot in enumerate(want):
                assert a[slot].tolist() == [bucket_start[s] + j, s]


# ------------------------------------------------------------------ element-wise parity

def test_tiny_full_size(torch_cuda):
    w = synth.make("tiny")
    gpu, orc = run_both(torch_cuda, w.ref, w.query, w.matrix, w.xdrop, w.K)
    assert gpu.total_hits > 30_000 and gpu.n_survivors > 10_000
    assert_same_as_oracle(gpu, orc)


@pytest.mark.parametrize("name,scale", [("mid", 0.1), ("dense", 0.03), ("workload_a", 0.02), ("chunking", 0.02)])
def test_scaled_workloads(torch_cuda, name, scale):
    w = synth.make(name, scale=scale)
    for qry in w.queries:
        gpu, orc = run_both(torch_cuda, w.ref, qry, w.matrix, w.xdrop, w.K, max_hits=w.max_hits)
        assert_same_as_oracle(gpu, orc)
        if name == "chunking":
            assert len(gpu.chunks) > 3


def test_chunk_walk_modes_agree(torch_cuda):
    w = synth.make("chunking", scale=0.02)
    a, orc = run_both(torch_cuda, w.ref, w.query, w.matrix, w.xdrop, w.K, max_hits=w.max_hits, walk_full=True)
    assert_same_as_oracle(a, orc)


def test_release_cached_memory_between_runs(torch_cuda):
    """Trimming the library's memory pools between two runs changes nothing."""
    from seed_hits_ungapped_gb300 import hspz
    w = synth.make("chunking", scale=0.02)
    eng = _engine(torch_cuda, w.ref, w.matrix, w.xdrop, w.K)
    a = eng.run(_dev(torch_cuda, w.query), max_hits=w.max_hits, keep=True)
    hspz.hspz_release_cached_memory()
    b = eng.run(_dev(torch_cuda, w.query), max_hits=w.max_hits, keep=True)
    for x, y in zip(a.per_chunk, b.per_chunk):
        assert np.array_equal(x.flags, y.flags) and np.array_equal(x.records, y.records)


def test_run_fetch_returns_every_chunk(torch_cuda):
    """fetch=True (the results-only copy the end-to-end timing uses) hands
    back each chunk's own records, done flags and accepted ids."""
    w = synth.make("chunking", scale=0.02)
    eng = _engine(torch_cuda, w.ref, w.matrix, w.xdrop, w.K)
    got = eng.run(_dev(torch_cuda, w.query), max_hits=w.max_hits, fetch=True)
    orc = oracle.run_path(w.ref, w.query, w.matrix, w.xdrop, w.K, max_hits=w.max_hits)
    assert len(got.per_chunk) == len(orc["per_chunk"]) > 3
    for g, o in zip(got.per_chunk, orc["per_chunk"]):
        assert g.anchors is None and g.flags is None
        assert np.array_equal(g.records, o["rec"])
        assert np.array_equal(g.done, o["done"])
        assert np.array_equal(g.accepted, o["accepted"])


@pytest.mark.parametrize("xdrop,K", [(0, 1), (50, 200), (910, 3000), (1 << 30, 5000)])
def test_general_matrix(torch_cuda, xdrop, K):
    """An asymmetric random matrix (not complement-symmetric) and extreme X/K."""
    rng = np.random.default_rng(xdrop + K)
    m = rng.integers(-150, 120, (5, 5)).astype(np.int32)
    m[np.arange(4), np.arange(4)] = rng.integers(60, 130, 4)
    w = synth.make("tiny", scale=0.2)
    gpu, orc = run_both(torch_cuda, w.ref, w.query, m, xdrop, K)
    assert_same_as_oracle(gpu, orc)


@pytest.mark.parametrize("xdrop,K", [(0, 1), (150, 600), (699, 2000), (700, 2000), (910, 3000), (910, 800)])
@pytest.mark.parametrize("name,scale", [("tiny", 0.2), ("mid", 0.02)])
def test_fast_gate_both_step_tests(torch_cuda, name, scale, xdrop, K):
    """HOXD70 (largest pair score 100) on both sides of X = 7 * 100: below it
    the 8-base step flags possible stops and replays them base by base, from
    it up the step's stop test is exact.  mid holds N runs."""
    w = synth.make(name, scale=scale)
    gpu, orc = run_both(torch_cuda, w.ref, w.query, w.matrix, xdrop, K)
    assert_same_as_oracle(gpu, orc)
    # the standalone round gate on the same anchors
    from seed_hits_ungapped_gb300 import hspz
    eng = _engine(torch_cuda, w.ref, w.matrix, xdrop, K)
    plan = eng.plan(_dev(torch_cuda, w.query))
    for g in gpu.per_chunk:
        anchors = torch_cuda.from_numpy(g.anchors.view(np.int32)).cuda()
        flags = torch_cuda.zeros(len(g.anchors), dtype=torch_cuda.uint8, device="cuda")
        hspz.hspz_score_gate_plan(eng.index, plan, anchors, len(g.anchors), eng.params, flags)
        assert np.array_equal(flags.cpu().numpy(), g.flags)
    plan.close()


@pytest.mark.parametrize("xdrop", [889, 888, 2000])
def test_fast_gate_int8_extreme_matrix(torch_cuda, xdrop):
    """The table-scored path with pair scores at the ends of int8 (A/T match
    +127, C/G match +120, transitions -60, transversions -128, N -100):
    exact 8-base stop test from X = 7 * 127 = 889 up, base-by-base replay
    below; every output equal to the oracle (mid scaled: N runs in both
    sequences)."""
    m = np.full((5, 5), -128, dtype=np.int32)
    for r, q in ((0, 2), (2, 0), (1, 3), (3, 1)):
        m[r, q] = -60
    m[0, 0] = m[3, 3] = 127
    m[1, 1] = m[2, 2] = 120
    m[4, :] = m[:, 4] = -100
    assert all(m[r, q] == m[r ^ 3, q ^ 3] for r in range(4) for q in range(4))  # complement symmetric
    w = synth.make("mid", scale=0.1)
    gpu, orc = run_both(torch_cuda, w.ref, w.query, m, xdrop, 3000, max_hits=20_000)
    flags = np.concatenate([pc["flags"] for pc in orc["per_chunk"]])
    assert 0 < flags.sum() < flags.size
    assert_same_as_oracle(gpu, orc)


def test_edges(torch_cuda):
    rng = np.random.default_rng(11)
    m = synth.hoxd70()
    s = rng.integers(0, 4, 5000).astype(np.uint8)
    # identical sequences: every anchor extends to both sequence edges
    gpu, orc = run_both(torch_cuda, s, s.copy(), m, 910, 3000)
    assert_same_as_oracle(gpu, orc)
    assert any((g.records[:, 0] == 0).any() for g in gpu.per_chunk)
    # query with N everywhere, a query shorter than the seed, an N-rich reference
    for qry in (np.full(400, 4, np.uint8), s[:18].copy(), s[:19].copy()):
        gpu, orc = run_both(torch_cuda, s, qry, m, 910, 3000)
        assert_same_as_oracle(gpu, orc)
    ref = s.copy()
    ref[rng.random(ref.size) < 0.2] = 4
    gpu, orc = run_both(torch_cuda, ref, s[1000:3000].copy(), m, 910, 3000)
    assert_same_as_oracle(gpu, orc)
    # a reference shorter than the seed span: an empty index
    gpu, orc = run_both(torch_cuda, s[:10].copy(), s[:500].copy(), m, 910, 3000)
    assert gpu.total_hits == 0 and orc["total"] == 0


def test_xdrop_and_threshold_extremes(torch_cuda):
    """Degenerate scoring parameters, everything equal to the oracle: X = 0
    (a walk stops at its first fall below its maximum; the 8-base stop test
    is not exact there), K = 1 (the keep threshold every anchor with a
    positive side reaches, so nearly every flag is set and the compactions
    see dense flags) and a threshold no anchor reaches (nothing survives)."""
    w = synth.make("tiny", scale=0.2)
    seen = {}
    for xdrop, K in ((0, 3000), (910, 1), (0, 1), (910, 10 ** 7)):
        gpu, orc = run_both(torch_cuda, w.ref, w.query, w.matrix, xdrop, K, max_hits=3000)
        assert_same_as_oracle(gpu, orc)
        flags = np.concatenate([pc["flags"] for pc in orc["per_chunk"]])
        seen[(xdrop, K)] = flags.mean()
    assert seen[(910, 1)] > 0.95 and seen[(910, 10 ** 7)] == 0.0
    assert seen[(0, 1)] > 0.5


@pytest.mark.parametrize("pattern,scale,max_hits", [
    ("11111111111", 0.2, 0),                                  # contiguous 11-mer
    ("111010010100110111", 0.2, 0),                           # another spaced seed
    ("1101011", 0.05, 100_000),                               # weight 5: ~50 hits per seed, chunked
    ("11100000000000000000000000000111", 0.2, 400_000),       # the longest span (32), weight 6
])
def test_other_seed_patterns(torch_cuda, pattern, scale, max_hits):
    """C.1-E.5 with seed patterns other than 12of19 (any weight up to 12 and
    span up to 32 is accepted): index, counts, prefix, chunks, anchors,
    flags, survivors and records all equal the oracle's."""
    w = synth.make("tiny", scale=scale)
    gpu, orc = run_both(torch_cuda, w.ref, w.query, w.matrix, w.xdrop, w.K, max_hits=max_hits, pattern=pattern)
    assert orc["total"] > 0
    assert_same_as_oracle(gpu, orc)


def test_expansion_mappings_and_standalone_gate(torch_cuda):
    """C.4: sparse and dense mappings give the fused kernel's anchors; the
    standalone gate over those anchors gives the fused flags."""
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    w = synth.make("dense", scale=0.03)
    eng = _engine(torch, w.ref, w.matrix, w.xdrop, w.K)
    plan = eng.plan(_dev(torch, w.query))
    n = plan.total_hits
    assert n > 100_000
    fused = torch.empty((n, 2), dtype=torch.int32, device="cuda")
    flags = torch.empty(n, dtype=torch.uint8, device="cuda")
    hspz.hspz_expand_gate(plan, 0, eng.params, fused, flags)
    for mode in (hspz.HSPZ_EXPAND_SPARSE, hspz.HSPZ_EXPAND_DENSE, hspz.HSPZ_EXPAND_AUTO):
        a = torch.full((n, 2), -1, dtype=torch.int32, device="cuda")
        hspz.hspz_expand(plan, 0, a, mode)
        assert torch.equal(a, fused)
    f2 = torch.full((n,), 7, dtype=torch.uint8, device="cuda")
    hspz.hspz_score_gate_plan(eng.index, plan, fused, n, eng.params, f2)
    assert torch.equal(f2, flags)


def test_compaction_alignment_and_capacity(torch_cuda):
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    rng = np.random.default_rng(5)
    for n in (1, 15, 16, 17, 4095, 4096, 4097, 100_003):
        f = (rng.random(n + 3) < 0.3).astype(np.uint8) * rng.integers(1, 256, n + 3).astype(np.uint8)
        d = torch.from_numpy(f).cuda()
        for off in (0, 1, 3):
            view = d[off:off + n]
            ids = torch.empty(n + 1, dtype=torch.int32, device="cuda")
            k = hspz.hspz_compact(view, n, 1000, ids)
            want = oracle.compact(f[off:off + n], 1000)
            assert k == want.size
            assert np.array_equal(ids[:k].cpu().numpy().view(np.uint32), want)
    # too small: nothing written, the needed count is reported
    f = np.ones(100, np.uint8)
    ids = torch.full((10,), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(hspz.HspzError) as e:
        hspz.hspz_compact(torch.from_numpy(f).cuda(), 100, 0, ids)
    assert e.value.needed == 100
    assert (ids.cpu().numpy() == -7).all()


def test_refusal_edge_on_gpu(torch_cuda):
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    ref = np.zeros(65_554, np.uint8)
    index = hspz.hspz_build_index(_dev(torch, ref))
    with pytest.raises(hspz.HspzError) as e:
        hspz.hspz_find_hits(index, _dev(torch, np.zeros(65_554, np.uint8)))
    assert e.value.status == hspz.HSPZ_E_HIT_OVERFLOW and e.value.total_hits == 1 << 32
    qry = np.zeros(65_553, np.uint8)
    cap = 1 << 30
    plan = hspz.hspz_find_hits(index, _dev(torch, qry), max_hits=cap)
    assert plan.total_hits == (1 << 32) - 65_536
    idx, pos = oracle.build_index(ref)
    P, total, rc = oracle.inclusive_prefix(oracle.count_hits(idx, oracle.seed_buckets(qry)))
    assert np.array_equal(plan.chunks, oracle.chunk_walk(P, cap))
    assert np.array_equal(plan.prefix().cpu().numpy().view(np.uint32), P)


# ------------------------------------------------------------------ full size, sampled

@pytest.mark.slow
def test_workload_a_full_size_sampled(torch_cuda):
    """The benchmark workload at full size, in the benchmark's launch
    configuration: full prefix, sampled anchors and flags, every survivor's
    flag, sampled records."""
    torch = torch_cuda
    w = synth.make("workload_a")
    eng = _engine(torch, w.ref, w.matrix, w.xdrop, w.K)
    gpu = eng.run(_dev(torch, w.query), keep=True)
    idx, pos = oracle.build_index(w.ref)
    buckets = oracle.seed_buckets(w.query)
    P, total, rc = oracle.inclusive_prefix(oracle.count_hits(idx, buckets))
    assert rc == 0 and gpu.total_hits == total
    assert np.array_equal(gpu.prefix, P)
    assert np.array_equal(gpu.chunks, oracle.chunk_walk(P, 0))
    ch = gpu.per_chunk[0]
    rng = np.random.default_rng(0)
    sample = np.unique(rng.integers(0, total, 20_000))
    want = oracle.anchors_at(idx, pos, buckets, P, sample)
    assert np.array_equal(ch.anchors[sample], want)
    assert np.array_equal(ch.flags[sample], oracle.gate(w.ref, w.query, want, w.matrix, w.xdrop, eng.T))
    # every survivor really passes, and survivors are exactly the set flags
    assert np.array_equal(ch.ids, np.flatnonzero(ch.flags).astype(np.uint32))
    assert oracle.gate(w.ref, w.query, ch.anchors[ch.ids], w.matrix, w.xdrop, eng.T).all()
    pick = np.unique(rng.integers(0, ch.ids.size, 5_000))
    rec, done = oracle.materialize(w.ref, w.query, ch.anchors, 0, ch.ids[pick], w.matrix, w.xdrop, eng.T)
    assert np.array_equal(ch.records[pick], rec) and np.array_equal(ch.done[pick], done)


@pytest.mark.parametrize("name,scale", [("workload_a", 0.02), ("mid", 0.1), ("dense", 0.03)])
def test_reference_bucketed_gate_equals_fused(torch_cuda, name, scale):
    """D.5: bucketing by reference window leaves every flag unchanged."""
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    w = synth.make(name, scale=scale)
    eng = _engine(torch, w.ref, w.matrix, w.xdrop, w.K)
    plan = eng.plan(_dev(torch, w.query))
    n = plan.total_hits
    anchors = torch.empty((n, 2), dtype=torch.int32, device="cuda")
    fused = torch.empty(n, dtype=torch.uint8, device="cuda")
    hspz.hspz_expand_gate(plan, 0, eng.params, anchors, fused)
    want = oracle.gate(w.ref, w.query, anchors.cpu().numpy().view(np.uint32), w.matrix, w.xdrop, eng.T)
    assert np.array_equal(fused.cpu().numpy(), want)
    for nb in (0, 1, 3, 32):
        got = torch.full((n,), 9, dtype=torch.uint8, device="cuda")
        hspz.hspz_score_gate_bucketed(eng.index, plan, anchors, n, eng.params, got, n_buckets=nb)
        assert torch.equal(got, fused), nb
    bad = hspz.score_params(np.arange(25).reshape(5, 5) - 12, w.xdrop, w.K)  # not complement symmetric
    with pytest.raises(hspz.HspzError):
        hspz.hspz_score_gate_bucketed(eng.index, plan, anchors, n, bad, fused)


def test_process_chunk_capacity_and_counts(torch_cuda):
    """hspz_process_chunk: too little survivor room is reported (anchors and
    flags written, survivor outputs untouched); with room it matches the
    oracle's survivors, records and accepted indices."""
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    w = synth.make("tiny", scale=0.3)
    eng = _engine(torch, w.ref, w.matrix, w.xdrop, w.K)
    plan = eng.plan(_dev(torch, w.query))
    n = plan.total_hits
    anchors = torch.empty((n, 2), dtype=torch.int32, device="cuda")
    flags = torch.empty(n, dtype=torch.uint8, device="cuda")
    small = [torch.full((4,), -3, dtype=torch.int32, device="cuda"), torch.full((4, 4), -3, dtype=torch.int32, device="cuda"),
             torch.full((4,), 9, dtype=torch.uint8, device="cuda"), torch.full((4,), -3, dtype=torch.int32, device="cuda")]
    with pytest.raises(hspz.HspzError) as e:
        hspz.hspz_process_chunk(plan, 0, eng.params, anchors, flags, *small)
    orc = oracle.run_path(w.ref, w.query, w.matrix, w.xdrop, w.K)["per_chunk"][0]
    assert e.value.needed == orc["ids"].size > 4
    assert (small[0].cpu().numpy() == -3).all() and (small[2].cpu().numpy() == 9).all()
    assert np.array_equal(flags.cpu().numpy(), orc["flags"])
    m = e.value.needed
    big = [torch.empty(m, dtype=torch.int32, device="cuda"), torch.empty((m, 4), dtype=torch.int32, device="cuda"),
           torch.empty(m, dtype=torch.uint8, device="cuda"), torch.empty(m, dtype=torch.int32, device="cuda")]
    ns, na, ms = hspz.hspz_process_chunk(plan, 0, eng.params, anchors, flags, *big, time_gate=True)
    assert ns == m and na == orc["accepted"].size and ms > 0
    assert np.array_equal(big[0].cpu().numpy().view(np.uint32), orc["ids"])
    assert np.array_equal(big[1].cpu().numpy(), orc["rec"])
    assert np.array_equal(big[2].cpu().numpy(), orc["done"])
    assert np.array_equal(big[3][:na].cpu().numpy().view(np.uint32), orc["accepted"])


def test_process_chunk_ragged_unaligned_short(torch_cuda):
    """hspz_process_chunk (C.5 through E.5 with the D.4 compactions) on chunks
    of ragged sizes, with the flag buffer at an odd address (the byte-load
    path of the compaction) and with a survivor buffer one slot short of the
    count (capacity error with the needed count)."""
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    w = synth.make("tiny", scale=0.3)
    max_hits = 1000
    eng = _engine(torch, w.ref, w.matrix, w.xdrop, w.K)
    plan = eng.plan(_dev(torch, w.query), max_hits)
    orc = oracle.run_path(w.ref, w.query, w.matrix, w.xdrop, w.K, max_hits=max_hits)
    assert np.array_equal(plan.chunks, orc["chunks"]) and len(orc["per_chunk"]) > 3
    sizes = set()
    for ci, pc in enumerate(orc["per_chunk"]):
        n = pc["flags"].size
        sizes.add(n % 256)
        anchors = torch.empty((n, 2), dtype=torch.int32, device="cuda")
        flags = torch.full((n + 1,), 7, dtype=torch.uint8, device="cuda")[1:]
        m = pc["ids"].size
        bufs = [torch.full((m + 1,), -3, dtype=torch.int32, device="cuda"),
                torch.empty((m + 1, 4), dtype=torch.int32, device="cuda"),
                torch.empty(m + 1, dtype=torch.uint8, device="cuda"),
                torch.empty(m + 1, dtype=torch.int32, device="cuda")]
        ns, na, _ = hspz.hspz_process_chunk(plan, ci, eng.params, anchors, flags, *bufs)
        assert ns == m and na == pc["accepted"].size
        assert np.array_equal(flags.cpu().numpy(), pc["flags"])
        assert np.array_equal(bufs[0][:m].cpu().numpy().view(np.uint32), pc["ids"])
        assert int(bufs[0][m]) == -3
        assert np.array_equal(bufs[1][:m].cpu().numpy(), pc["rec"])
        if m:
            short = [b[:m - 1] for b in bufs]
            with pytest.raises(hspz.HspzError) as e:
                hspz.hspz_process_chunk(plan, ci, eng.params, anchors, flags, *short)
            assert e.value.needed == m
    assert len(sizes) > 1  # chunk ends fall at different places of a 256-anchor block


def test_materialize_any_id_order(torch_cuda):
    """E.1-E.5 per survivor, whatever the id list: ascending survivors (long
    runs of neighbours on one diagonal), reversed, shuffled, with duplicates,
    with ids outside the anchors, every anchor of a chunk, and lists cut so
    that runs start and end at every place; in list order and in diagonal
    order (grouped).  Each record must equal the oracle's record for that id
    alone, at that id's place."""
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    rng = np.random.default_rng(23)
    m = synth.hoxd70()
    s = rng.integers(0, 4, 6000).astype(np.uint8)
    ref = s.copy()
    ref[2500:2510] = 4                        # N inside the long diagonal
    qry = np.concatenate([s[1000:4000], rng.integers(0, 4, 500).astype(np.uint8), s[4000:5200]])
    qry[rng.random(qry.size) < 0.06] = rng.integers(0, 4, 1).astype(np.uint8)
    w = synth.make("tiny")
    for r, q in ((ref, qry), (w.ref, w.query)):
        eng = _engine(torch, r, m, 910, 3000)
        plan = eng.plan(_dev(torch, q))
        n = plan.total_hits
        anchors = torch.empty((n, 2), dtype=torch.int32, device="cuda")
        flags = torch.empty(n, dtype=torch.uint8, device="cuda")
        hspz.hspz_expand_gate(plan, 0, eng.params, anchors, flags)
        a_np = anchors.cpu().numpy().view(np.uint32)
        surv = np.nonzero(flags.cpu().numpy())[0].astype(np.int64)
        base = 77
        lists = [surv, surv[::-1], rng.permutation(surv), np.repeat(surv[:300], 2),
                 np.arange(n), np.concatenate([surv[:50], [n + 5, n + 6], surv[50:120], [0], surv[120:]])]
        lists += [surv[c:] for c in (1, 7, 131)] + [surv[:c] for c in (1, 2, 9, 200)]
        for ids_local in lists:
            ids = (np.asarray(ids_local, np.int64) + base).astype(np.uint32)
            k = ids.size
            d_ids = torch.from_numpy(ids.view(np.int32)).cuda()
            # an id outside the anchors gets an empty record (the oracle takes valid ids only)
            valid = np.asarray(ids_local, np.int64) < n
            rec_o = np.zeros((k, 4), np.int32)
            done_o = np.zeros(k, np.uint8)
            rec_o[valid], done_o[valid] = oracle.materialize(r, q, a_np, base, ids[valid], m, 910, 3000)
            for grouped in (False, True):
                out = torch.full((max(k, 1), 4), -3, dtype=torch.int32, device="cuda")
                done = torch.full((max(k, 1),), 9, dtype=torch.uint8, device="cuda")
                hspz.hspz_materialize_plan(eng.index, plan, anchors, base, d_ids, k, eng.params, out, done,
                                      grouped=grouped)
                assert np.array_equal(done[:k].cpu().numpy(), done_o)
                assert np.array_equal(out[:k].cpu().numpy(), rec_o)


def test_run_stream_batches_match_oracle(torch_cuda):
    """HspEngine.run_stream: uploads and result copies on a copy stream,
    overlapping the next batch.  Every batch, chunk by chunk, must hold the
    oracle's records, done flags and accepted ids; several chunks per batch
    (MAX_HITS cuts) make the two result sets alternate within a batch.  A
    consumer that stops early leaves the engine usable."""
    torch = torch_cuda
    w = synth.make("tiny")
    m = w.matrix
    eng = _engine(torch, w.ref, m, w.xdrop, w.K)
    qs = [w.query, w.query[:60_000].copy(), w.query[:12].copy(), w.query[::-1].copy(), w.query[100_000:].copy()]
    pinned = [torch.from_numpy(np.ascontiguousarray(q)).pin_memory() for q in qs]
    for max_hits in (0, 4000):
        got = 0
        for q, res in zip(qs, eng.run_stream(pinned, max_hits=max_hits)):
            orc = oracle.run_path(w.ref, q, m, w.xdrop, w.K, max_hits=max_hits)
            assert res.total_hits == orc["total"]
            assert len(res.per_chunk) == len(orc["per_chunk"])
            for g, o in zip(res.per_chunk, orc["per_chunk"]):
                assert np.array_equal(g.records, o["rec"])
                assert np.array_equal(g.done, o["done"])
                assert np.array_equal(g.accepted, o["accepted"])
            got += 1
        assert got == len(qs)
    gen = eng.run_stream(pinned, max_hits=0)
    next(gen)
    gen.close()  # the second batch's upload was already under way
    res = next(eng.run_stream(pinned[1:2], max_hits=0))
    orc = oracle.run_path(w.ref, qs[1], m, w.xdrop, w.K)
    assert res.total_hits == orc["total"]
    assert all(np.array_equal(g.records, o["rec"]) for g, o in zip(res.per_chunk, orc["per_chunk"]))


def test_repetitive_chunks_group_by_diagonal(torch_cuda):
    """Poly-A and (CA)n repeats: one seed hits many reference positions, so a
    chunk averages >= 64 hits per seed and an engine with group=True
    materializes it in diagonal order (hspz_materialize_grouped).  Everything
    must still equal the oracle, with and without MAX_HITS cuts, and with
    grouping off."""
    torch = torch_cuda
    rng = np.random.default_rng(41)
    m = synth.hoxd70()
    ref = rng.integers(0, 4, 30_000).astype(np.uint8)
    ref[5_000:5_600] = 0                                   # poly-A
    for i in range(12):                                    # (CA)n copies
        p0 = 8_000 + 1_500 * i
        ref[p0:p0 + 160] = np.tile(np.array([1, 0], np.uint8), 80)
    qry = rng.integers(0, 4, 3_000).astype(np.uint8)
    qry = np.concatenate([qry[:1_000], np.zeros(500, np.uint8), qry[1_000:2_000],
                          np.tile(np.array([1, 0], np.uint8), 120), qry[2_000:]])
    qry[1_200] = 2                                          # a mismatch inside the poly-A run
    for max_hits, group in ((0, True), (60_000, True), (0, False)):
        from seed_hits_ungapped_gb300.engine import HspEngine
        eng = HspEngine(ref, m, 910, 3000, group=group)
        plan = eng.plan(_dev(torch, qry), max_hits)
        if group:
            assert any(eng.chunk_is_repetitive(plan, c) for c in range(plan.n_chunks))
        plan.close()
        gpu = eng.run(_dev(torch, qry), max_hits=max_hits, keep=True)
        orc = oracle.run_path(ref, qry, m, 910, 3000, max_hits=max_hits)
        assert_same_as_oracle(gpu, orc)
        assert gpu.n_survivors > 10_000
