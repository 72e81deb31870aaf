"""The gate and the materializer on raw device sequences (hspz_score_gate,
hspz_materialize: "D. Score gate" D.1-D.3 and "E. X-drop materialization"
E.1-E.5 with anchors and encoded sequences as the only inputs), through the
C ABI, against the oracle's gate and materialization element by element.

Anchors come from three places: the seed hits of the path itself, random
coordinates (not seed matches, so walks start anywhere, also next to the
sequence edges), and coordinates outside the sequences (flag 0, rejected
slot).  The matrices cover the fast table with the exact 8-base stop test
(HOXD70, X = 910), the fast table with replayed steps (X = 600) and an
asymmetric matrix the fast table cannot hold; the sequences hold N runs.
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


def _asymmetric():
    rng = np.random.default_rng(31)
    m = rng.integers(-140, 60, (5, 5)).astype(np.int32)
    m[np.arange(4), np.arange(4)] = rng.integers(70, 120, 4)
    return m


def _anchors(w, rng):
    res = oracle.run_path(w.ref, w.query, w.matrix, w.xdrop, w.K)
    seeds = np.concatenate([pc["anchors"] for pc in res["per_chunk"]])
    Lr, Lq = w.ref.size, w.query.size
    rand = np.stack([rng.integers(0, Lr, 3000), rng.integers(0, Lq, 3000)], 1)
    edges = np.array([[0, 0], [Lr - 1, Lq - 1], [0, Lq - 1], [Lr - 1, 0], [1, 1], [7, 9], [Lr - 8, Lq - 3]])
    inside = np.concatenate([seeds.astype(np.int64), rand, edges]).astype(np.uint32)
    outside = np.array([[Lr, 0], [0, Lq], [Lr + 5, Lq + 5], [0xFFFFFFFF, 3], [3, 0xFFFFFFFF]], np.uint32)
    a = np.concatenate([inside, outside])
    perm = rng.permutation(a.shape[0])
    return a[perm], perm < inside.shape[0]


@pytest.mark.parametrize("which", ["hoxd70_exact", "hoxd70_replay", "asymmetric"])
def test_raw_gate_and_materialize_match_oracle(torch_cuda, which):
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    rng = np.random.default_rng(5)
    w = synth.make("mid", scale=0.02)
    m, X, K = {"hoxd70_exact": (w.matrix, 910, 3000), "hoxd70_replay": (w.matrix, 600, 2000),
               "asymmetric": (_asymmetric(), 500, 900)}[which]
    a, inside = _anchors(w, rng)
    n = a.shape[0]
    T = oracle.keep_threshold(K)
    want = np.zeros(n, np.uint8)
    want[inside] = oracle.gate(w.ref, w.query, a[inside], m, X, T)
    assert 0 < want.sum() < inside.sum()
    d_ref = torch.from_numpy(w.ref).cuda()
    d_qry = torch.from_numpy(w.query).cuda()
    d_a = torch.from_numpy(a.view(np.int32)).cuda()
    flags = torch.full((n,), 7, dtype=torch.uint8, device="cuda")
    params = hspz.score_params(m, X, K)
    hspz.hspz_score_gate(d_a, n, d_ref, d_qry, params, flags)
    assert np.array_equal(flags.cpu().numpy(), want)

    # materialize: the survivors, some rejected anchors, ids outside the anchor array
    base = 1000
    surv = np.flatnonzero(want)
    rej = np.flatnonzero(inside & (want == 0))[:200]
    outs = np.flatnonzero(~inside)
    ids_local = np.concatenate([surv, rej, outs, [n, n + 3]])
    ids_local = ids_local[rng.permutation(ids_local.size)]
    ids = (ids_local + base).astype(np.uint32)
    k = ids.size
    rec_o = np.zeros((k, 4), np.int32)
    done_o = np.zeros(k, np.uint8)
    ok = (ids_local < n) & np.concatenate([inside, [False]])[np.minimum(ids_local, n)]
    rec_o[ok], done_o[ok] = oracle.materialize(w.ref, w.query, a, base, ids[ok], m, X, T)
    out = torch.full((k, 4), -3, dtype=torch.int32, device="cuda")
    done = torch.full((k,), 9, dtype=torch.uint8, device="cuda")
    hspz.hspz_materialize(d_a, base, torch.from_numpy(ids.view(np.int32)).cuda(), k, d_ref, d_qry, params, out, done)
    assert np.array_equal(done.cpu().numpy(), done_o)
    assert np.array_equal(out.cpu().numpy(), rec_o)
    assert done_o.sum() == surv.size  # every survivor is accepted (done = score >= T)


@pytest.mark.parametrize("X", [910, 600])
def test_walks_past_2_pow_20_steps_match_oracle(torch_cuda, X):
    """E.2/E.3 on sides longer than 2^20 steps of 8 bases, where the 32-bit
    running sum of the 8-base walk hands the survivor over to the 64-bit
    base-by-base walk: 17 Mbp sequences that agree everywhere but at a few
    scattered bases, anchors in the middle (both sides ~8.5 Mbp), near the
    start (right side ~17 Mbp) and on one diagonal a few bases apart (joined
    walks), with the exact 8-base stop test (X = 910) and the replayed one
    (X = 600).  Records and flags equal the oracle's."""
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    rng = np.random.default_rng(77)
    L = 17_000_000
    ref = rng.integers(0, 4, L).astype(np.uint8)
    qry = ref.copy()
    mis = rng.choice(L, 40, replace=False)
    qry[mis] = (qry[mis] + 1) % 4
    m, K = synth.hoxd70(), 3000
    T = oracle.keep_threshold(K)
    a = np.array([[L // 2, L // 2], [L // 2 + 37, L // 2 + 37], [100, 100], [L - 50, L - 50]], np.uint32)
    d_ref, d_qry = torch.from_numpy(ref).cuda(), torch.from_numpy(qry).cuda()
    d_a = torch.from_numpy(a.view(np.int32)).cuda()
    params = hspz.score_params(m, X, K)
    flags = torch.full((a.shape[0],), 7, dtype=torch.uint8, device="cuda")
    hspz.hspz_score_gate(d_a, a.shape[0], d_ref, d_qry, params, flags)
    assert np.array_equal(flags.cpu().numpy(), oracle.gate(ref, qry, a, m, X, T))
    ids = np.arange(a.shape[0], dtype=np.uint32)
    rec_o, done_o = oracle.materialize(ref, qry, a, 0, ids, m, X, T)
    assert rec_o[0, 2] > 8 * (1 << 21)  # both sides of the middle anchor pass 2^20 steps
    out = torch.full((ids.size, 4), -3, dtype=torch.int32, device="cuda")
    done = torch.full((ids.size,), 9, dtype=torch.uint8, device="cuda")
    hspz.hspz_materialize(d_a, 0, torch.from_numpy(ids.view(np.int32)).cuda(), ids.size, d_ref, d_qry, params, out,
                          done)
    assert np.array_equal(done.cpu().numpy(), done_o)
    assert np.array_equal(out.cpu().numpy(), rec_o)
