"""Pins for the CPU oracle: values fixed by the hspZ pages or by mathematics.

Nothing here re-types the oracle's own loops.  Each test checks the oracle
against something independent of it: the worked example printed in "C. Hit
discovery", brute-force enumeration, closed forms, textbook maximum prefix
sums, hand-computed cases, numpy's own f32 rounding, or invariants the pages
state in words.  Several cases use an asymmetric matrix so that a transposed
operand cannot hide behind a symmetric one.
"""
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
PATTERN = "1110100110010101111"
CARE = [i for i, c in enumerate(PATTERN) if c == "1"]
SPAN = len(PATTERN)
DIAG_HOXD70 = {0: 91, 1: 100, 2: 100, 3: 91}


def hoxd70():
    m = np.full((5, 5), -100, dtype=np.int32)
    m[:4, :4] = [[91, -114, -31, -123], [-114, 100, -125, -31], [-31, -125, 100, -114], [-123, -31, -114, 91]]
    return m


def _golden():
    rows = {}
    slots = {}
    with open(os.path.join(HERE, "golden", "hit_discovery_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            vals = [int(v) for v in vals]
            if key == "slots":
                slots[vals[0]] = vals[1:]
            else:
                rows[key] = vals
    return rows, slots


# ---------------------------------------------------------------- hit discovery

def _worked_index():
    """A 4-bucket index whose buckets hold 0, 3, 1 and 5 reference ends."""
    idx = np.array([0, 3, 4, 9], dtype=np.uint32)  # inclusive bucket ends
    pos = np.array([110, 111, 112, 220, 330, 331, 332, 333, 334], dtype=np.uint32)
    buckets = np.array([0, 1, 2, -1, 3], dtype=np.int64)  # seed 3 has no k-mer
    return idx, pos, buckets


def test_worked_example_counts_and_prefix():
    rows, _ = _golden()
    idx, pos, buckets = _worked_index()
    cnt = oracle.count_hits(idx, buckets)
    assert cnt.tolist() == rows["counts"]
    P, total, rc = oracle.inclusive_prefix(cnt)
    assert rc == 0
    assert P.tolist() == rows["prefix"]
    assert total == rows["prefix"][-1]


def test_worked_example_backward_slots():
    rows, slots = _golden()
    idx, pos, buckets = _worked_index()
    P = np.array(rows["prefix"], dtype=np.uint32)
    anchors = oracle.expand(idx, pos, buckets, P, [0, 5, 0, 9], span=SPAN)
    assert anchors.shape == (9, 2)
    for s, want in slots.items():
        start = int(idx[buckets[s] - 1]) if buckets[s] > 0 else 0
        for j, slot in enumerate(want):
            assert anchors[slot, 0] == pos[start + j]
            assert anchors[slot, 1] == s + SPAN - 1
    # a chunk that starts at seed 2 (hit 3) shifts every slot down by its start
    sub = oracle.expand(idx, pos, buckets, P, [2, 5, 3, 9], span=SPAN)
    full = anchors[3:9]
    assert np.array_equal(sub, full)
    # one by one
    one = oracle.anchors_at(idx, pos, buckets, P, range(9), span=SPAN)
    assert np.array_equal(one, anchors)


def _kmer_match(ref, qry, r, q):
    for c in CARE:
        a, b = ref[r + c], qry[q + c]
        if a > 3 or b > 3 or a != b:
            return False
    return True


def _low_complexity(rng, n, n_frac=0.01):
    s = rng.choice(np.array([0, 1], dtype=np.uint8), size=n, p=[0.6, 0.4])
    s[rng.random(n) < 0.03] = 2
    s[rng.random(n) < 0.02] = 3
    s[rng.random(n) < n_frac] = 4
    return s.astype(np.uint8)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_anchors_equal_brute_force_matches(seed):
    rng = np.random.default_rng(seed)
    ref = _low_complexity(rng, 500)
    qry = _low_complexity(rng, 260)
    qry[100:160] = ref[300:360]  # a planted copy
    pairs = [(r + SPAN - 1, q + SPAN - 1)
             for q in range(len(qry) - SPAN + 1)
             for r in range(len(ref) - SPAN + 1)
             if _kmer_match(ref, qry, r, q)]
    # raw order: query end ascending, and within a seed the reference end descending
    pairs.sort(key=lambda t: (t[1], -t[0]))
    assert len(pairs) > 20
    res = oracle.run_path(ref, qry, hoxd70(), 910, 3000)
    assert res["rc"] == 0
    assert res["total"] == len(pairs)
    got = res["per_chunk"][0]["anchors"]
    assert [tuple(map(int, a)) for a in got] == pairs
    per_seed = np.zeros(len(qry) - SPAN + 1, dtype=np.int64)
    for _, qe in pairs:
        per_seed[qe - SPAN + 1] += 1
    assert res["cnt"].tolist() == per_seed.tolist()


def test_index_lists_every_window_once_in_ascending_bucket_runs():
    rng = np.random.default_rng(7)
    ref = _low_complexity(rng, 400, n_frac=0.02)
    idx, pos = oracle.build_index(ref, PATTERN)
    windows = [r for r in range(len(ref) - SPAN + 1) if all(ref[r + c] < 4 for c in CARE)]
    assert sorted(pos.tolist()) == [r + SPAN - 1 for r in windows]
    assert int(idx[-1]) == len(windows)
    assert np.all(np.diff(idx.astype(np.int64)) >= 0)
    starts = np.concatenate([[0], idx[:-1]]).astype(np.int64)
    for h in np.flatnonzero(idx.astype(np.int64) - starts):
        run = pos[starts[h]:idx[h]]
        assert np.all(np.diff(run.astype(np.int64)) > 0)
        # every window in one bucket run shares its care bases
        r0 = int(run[0]) - SPAN + 1
        for e in run[1:]:
            assert _kmer_match(ref, ref, r0, int(e) - SPAN + 1)


def test_refusal_edge_at_2_pow_32():
    # all-A reference and query: every window of both falls in bucket 0.
    ref = np.zeros(65_554, dtype=np.uint8)
    # 65,536 reference windows x 65,536 query seeds = 2^32 hits: refused
    res = oracle.run_path(ref, np.zeros(65_554, dtype=np.uint8), hoxd70(), 910, 3000, max_hits=1 << 20,
                          index=oracle.build_index(ref))
    assert res["rc"] == oracle.ORC_E_OVERFLOW
    # one seed fewer: 2^32 - 65,536 hits, accepted (plan only)
    idx, pos = oracle.build_index(ref)
    b = oracle.seed_buckets(np.zeros(65_553, dtype=np.uint8))
    P, total, rc = oracle.inclusive_prefix(oracle.count_hits(idx, b))
    assert rc == 0 and total == (1 << 32) - 65_536


# ---------------------------------------------------------------- chunk walk

@pytest.mark.parametrize("seed", range(6))
def test_chunk_walk_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    S = int(rng.integers(1, 400))
    cnt = rng.integers(0, 9, S).astype(np.uint32)
    cnt[rng.random(S) < 0.4] = 0
    if seed == 0:
        cnt[-20:] = 0  # trailing zero-count seeds
    P, total, rc = oracle.inclusive_prefix(cnt)
    assert rc == 0
    for cap in sorted({1, 2, 3, 5, 8, 13, 40, max(1, total // 3), max(1, total), total + 1}):
        ch = oracle.chunk_walk(P, cap).astype(np.int64)
        assert ch[0, 0] == 0 and ch[-1, 1] == S and ch[0, 2] == 0 and ch[-1, 3] == total
        assert np.all(ch[1:, 0] == ch[:-1, 1]) and np.all(ch[1:, 2] == ch[:-1, 3])
        assert np.all(ch[:, 1] > ch[:, 0])
        for sb, se, hb, he in ch:
            assert hb == (int(P[sb - 1]) if sb else 0) and he == int(P[se - 1])  # no seed is split
        if total <= cap:
            assert len(ch) == 1
        for k, (sb, se, hb, he) in enumerate(ch):
            if k < len(ch) - 1:
                assert he - hb >= cap  # a cut chunk reaches the cap ...
                assert he - hb - int(cnt[se - 1]) < cap  # ... and overruns it by less than its last seed
            else:  # the last chunk either fits the cap or is cut at the last seed
                assert he - hb <= cap or he - hb - int(cnt[se - 1]) < cap
        # concatenated chunk expansions equal the unchunked stream
        idx = np.concatenate([[0], np.cumsum(np.arange(1, 10))]).astype(np.uint32)[1:]
        buckets = np.where(cnt > 0, cnt.astype(np.int64) - 1, -1)
        pos = np.arange(int(idx[-1]), dtype=np.uint32) * 7
        whole = oracle.expand(idx, pos, buckets, P, [0, S, 0, total])
        parts = [oracle.expand(idx, pos, buckets, P, c) for c in ch.astype(np.uint32)]
        assert np.array_equal(np.concatenate(parts) if parts else whole[:0], whole)


# ---------------------------------------------------------------- X-drop walks

def _seq(s):
    return np.array(["ACGTN".index(c) for c in s], dtype=np.uint8)


@pytest.mark.parametrize("a", [0, 1, 57, 298, 299])
def test_all_match_closed_form(a):
    rng = np.random.default_rng(a)
    s = rng.integers(0, 4, 300).astype(np.uint8)
    m = hoxd70()
    sc = oracle.side_scores(s, s, [[a, a]], m, 910)[0]
    left = sum(DIAG_HOXD70[int(b)] for b in s[:a])
    right = sum(DIAG_HOXD70[int(b)] for b in s[a:])
    assert sc.tolist() == [left, a, right, 300 - a]
    rec, done = oracle.materialize(s, s, [[a, a]], 0, [0], m, 910, 3000)
    assert rec[0].tolist() == [0, 0, 299, left + right] and done[0] == 1


@pytest.mark.parametrize("seed", range(8))
def test_infinite_xdrop_is_max_prefix_sum(seed):
    rng = np.random.default_rng(seed)
    L = 120
    ref = rng.integers(0, 5, L).astype(np.uint8)
    qry = np.where(rng.random(L) < 0.6, ref, rng.integers(0, 5, L)).astype(np.uint8)
    m = rng.integers(-60, 61, (5, 5)).astype(np.int32)  # asymmetric on purpose
    a = int(rng.integers(0, L))
    sc = oracle.side_scores(ref, qry, [[a, a]], m, 1 << 30)[0]
    # brute force over every (l, r) window [a-l, a+r) around the anchor
    best, arg = None, None
    for l in range(a + 1):
        for r in range(L - a + 1):
            tot = sum(int(m[ref[k], qry[k]]) for k in range(a - l, a + r))
            if best is None or tot > best:
                best, arg = tot, (l, r)
    assert sc[0] + sc[2] == best
    # the earliest maximum on each side is the smallest extent that attains it
    assert (sc[1], sc[3]) == arg


def _hand_matrix():
    m = np.full((5, 5), -100, dtype=np.int32)
    m[0, 0] = 10   # A/A
    m[0, 1] = -10  # ref A vs query C
    m[1, 0] = 40   # ref C vs query A: asymmetric on purpose
    m[2, 2] = 50   # G/G
    m[1, 1] = -25  # C/C
    m[3, 3] = -35  # T/T
    m[2, 3] = 100  # ref G vs query T
    return m


def test_drop_is_strictly_beyond_x():
    m = _hand_matrix()
    # right side from the anchor: +10, -10, -10, +50, then -100
    ref = _seq("T" + "AAAGT")
    qry = _seq("A" + "ACCGA")
    sc = oracle.side_scores(ref, qry, [[1, 1]], m, 20)[0]
    # S = 10, 0, -10 (deficit exactly X: the walk goes on), 40, -60 (stop)
    assert sc[2:].tolist() == [40, 4]
    sc = oracle.side_scores(ref, qry, [[1, 1]], m, 19)[0]
    assert sc[2:].tolist() == [10, 1]


def test_earliest_maximum_wins_on_ties():
    m = _hand_matrix()
    # right: +10, -10, +10 (ties the maximum later), then -100
    ref = _seq("T" + "AAAT")
    qry = _seq("A" + "ACAA")
    sc = oracle.side_scores(ref, qry, [[1, 1]], m, 500)[0]
    assert sc[2:].tolist() == [10, 1]
    # left mirror: bases before the anchor at 4 are (from the anchor outward) +10, -10, +10, -100
    ref = _seq("TAAA" + "T")
    qry = _seq("AACA" + "A")
    sc = oracle.side_scores(ref, qry, [[4, 4]], m, 500)[0]
    assert sc[:2].tolist() == [10, 1]
    rec, done = oracle.materialize(ref, qry, [[4, 4]], 0, [0], m, 500, 5)
    assert rec[0].tolist() == [3, 3, 0, 10] and done[0] == 1


def test_anchor_base_belongs_to_the_right_side():
    m = _hand_matrix()
    # right side, anchor base included: C/C -25, T/T -35, ref G/query T +100, ref A/query C -10
    ref = _seq("AC" + "CTG" + "A")
    qry = _seq("CC" + "CTT" + "C")
    sc = oracle.side_scores(ref, qry, [[2, 2]], m, 70)[0]
    # right: S = -25, -60 (deficit 60 <= 70), +40 -> max 40 at 3 bases; then ref A/qry C -10 -> 30
    # left: ref C/qry C -25 (deficit 25), then ref A/qry C -10 -> -35, edge: max 0
    assert sc.tolist() == [0, 0, 40, 3]
    # had the anchor base belonged to the left side the right maximum would be 65
    rec, done = oracle.materialize(ref, qry, [[2, 2]], 0, [0], m, 70, 40)
    assert rec[0].tolist() == [2, 2, 2, 40] and done[0] == 1


def test_matrix_rows_are_reference_bases():
    m = _hand_matrix()
    ref = _seq("C")
    qry = _seq("A")
    assert oracle.side_scores(ref, qry, [[0, 0]], m, 100)[0, 2] == 40
    assert oracle.side_scores(qry, ref, [[0, 0]], m, 100)[0, 2] == 0  # ref A vs query C is -10


def test_n_scores_by_matrix_and_edges_stop():
    m = hoxd70()
    ref = _seq("ACGNNACG")
    qry = _seq("ACGTAACG")
    sc = oracle.side_scores(ref, qry, [[0, 0]], m, 1000)[0]
    # right: 91, 100, 100, N/T -100, N/A -100, 91, 100, 100, then the sequence edge
    pref = np.cumsum([91, 100, 100, -100, -100, 91, 100, 100])
    assert sc[2] == pref.max() and sc[3] == int(np.argmax(pref)) + 1


# ---------------------------------------------------------------- threshold

def test_keep_threshold_matches_f32_compare():
    rng = np.random.default_rng(5)
    Ks = [1, 2, 3000, (1 << 24) - 1, 1 << 24, (1 << 24) + 1, (1 << 24) + 3, (1 << 25) + 5,
          123_456_789, (1 << 31) - 1] + rng.integers(1, 1 << 31, 40).tolist()
    for K in Ks:
        T = oracle.keep_threshold(K)
        assert 1 <= T <= K
        fK = np.float32(K)
        assert np.float32(T) >= fK
        assert T == 1 or np.float32(T - 1) < fK
        if K <= (1 << 24):
            assert T == K
    for K in range(1, 3000, 97):
        assert oracle.keep_threshold(K) == K
    with pytest.raises(oracle.OracleError):
        oracle.keep_threshold(0)


# ---------------------------------------------------------------- compaction / materialize

def test_compaction_is_stable_and_global():
    rng = np.random.default_rng(9)
    flags = (rng.random(10_001) < 0.03).astype(np.uint8)
    ids = oracle.compact(flags, 12345)
    assert np.array_equal(ids, np.flatnonzero(flags).astype(np.uint32) + 12345)
    assert oracle.compact(np.zeros(0, np.uint8)).size == 0


def test_materialized_records_score_their_closed_interval():
    from seed_hits_ungapped_gb300 import synth
    w = synth.make("tiny", scale=0.1)
    res = oracle.run_path(w.ref, w.query, w.matrix, w.xdrop, w.K)
    m = w.matrix
    seen = 0
    for ch in res["per_chunk"]:
        ids, rec, done = ch["ids"], ch["rec"], ch["done"]
        assert np.array_equal(ids, np.flatnonzero(ch["flags"]).astype(np.uint32) + int(res["chunks"][0][2]))
        sides = oracle.side_scores(w.ref, w.query, ch["anchors"][ids], m, w.xdrop)
        for k in range(ids.size):
            rs, qs, ln, score = map(int, rec[k])
            diag = [int(m[w.ref[rs + t], w.query[qs + t]]) for t in range(ln + 1)]
            assert sum(diag) == score == sides[k, 0] + sides[k, 2]
            assert done[k] == (score >= res["T"])
            a_r, a_q = map(int, ch["anchors"][ids[k]])
            assert a_r - rs == a_q - qs == sides[k, 1]  # the left extent shifts both starts
            assert ln + 1 == sides[k, 1] + sides[k, 3]
            seen += 1
    assert seen > 100


# ---------------------------------------------------------------- dedup (criterion: reading, parity unpinned)

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dedup_equals_pairwise_brute_force(seed):
    """keep[i] = 1 iff no earlier record equals record i in all four fields."""
    rng = np.random.default_rng(seed)
    n = 400
    rec = rng.integers(-2, 3, (n, 4)).astype(np.int32)
    rec[rng.random(n) < 0.1] = [np.iinfo(np.int32).min, np.iinfo(np.int32).max, 0, -1]
    keep = oracle.dedup(rec)
    for i in range(n):
        earlier = any((rec[j] == rec[i]).all() for j in range(i))
        assert keep[i] == (0 if earlier else 1)


def test_dedup_properties_and_edges():
    rng = np.random.default_rng(5)
    rec = rng.integers(0, 4, (5000, 4)).astype(np.int32)
    keep = oracle.dedup(rec).astype(bool)
    kept = rec[keep]
    # as many kept as there are distinct rows, all distinct, first occurrences
    assert kept.shape[0] == np.unique(rec, axis=0).shape[0]
    assert np.unique(kept, axis=0).shape[0] == kept.shape[0]
    _, first = np.unique(rec, axis=0, return_index=True)
    assert np.array_equal(np.sort(first), np.flatnonzero(keep))
    # records that differ in one field only, in the sign of a field, or not at all
    r = np.array([[1, 2, 3, 4], [1, 2, 3, -4], [1, 2, 3, 4], [0, 2, 3, 4], [1, 2, 3, 4]], np.int32)
    assert oracle.dedup(r).tolist() == [1, 1, 0, 1, 0]
    assert oracle.dedup(np.zeros((0, 4), np.int32)).size == 0
    assert oracle.dedup(np.ones((7, 4), np.int32)).tolist() == [1, 0, 0, 0, 0, 0, 0]


def test_dedup_leaves_one_hsp_per_exact_copy():
    """A query holding an exact 300 bp copy of the reference between N runs:
    every seed hit on that diagonal extends over the whole copy (all pair
    scores positive, the N flanks stop both sides after 10 bases), so all the
    accepted records are equal and dedup keeps exactly the first one, with
    the closed-form score of the copy."""
    rng = np.random.default_rng(21)
    m = hoxd70()
    ref = rng.integers(0, 4, 20_000).astype(np.uint8)
    seg = ref[7_000:7_300]
    qry = np.concatenate([np.full(50, 4, np.uint8), seg, np.full(50, 4, np.uint8)])
    res = oracle.run_path(ref, qry, m, 910, 3000)
    acc = res["accepted_rec"]
    assert acc.shape[0] > 100
    score = sum(DIAG_HOXD70[int(b)] for b in seg)
    assert res["final_rec"].tolist() == [[7_000, 50, 299, score]]
    assert res["final_idx"].tolist() == [0]


def _side_pairs_np(m, ref, qry, ar, aq, right, X, need):
    """Pairs a side walk scores, from prefix sums: the first n where the
    drop below the running maximum passes X, the maximum reaches `need`, or
    the sequence edge comes."""
    if right:
        r, q = ref[ar:], qry[aq:]
        k = min(r.size, q.size)
        sc = m[r[:k], q[:k]].astype(np.int64)
    else:
        k = min(ar, aq)
        sc = m[ref[ar - k:ar][::-1], qry[aq - k:aq][::-1]].astype(np.int64)
    if k == 0:
        return 0, 0
    S = np.cumsum(sc)
    Mrun = np.maximum.accumulate(np.maximum(S, 0))
    Mprev = np.concatenate([[0], Mrun[:-1]])
    ends = [k]
    drop = np.nonzero(Mprev - S > X)[0]
    if drop.size:
        ends.append(drop[0] + 1)
    acc = np.nonzero(Mrun >= need)[0]
    if acc.size:
        ends.append(acc[0] + 1)
    n = min(ends)
    best = int(Mprev[n - 1]) if (drop.size and n == drop[0] + 1) else int(Mrun[n - 1])
    return n, best


@pytest.mark.parametrize("T", [3000, 400, 10 ** 9])
def test_gate_pairs_matches_prefix_sum_form(T):
    rng = np.random.default_rng(17 + T % 1000)
    m = hoxd70()
    m[0, 2] = -60  # asymmetric, so a transposed lookup changes the count
    ref = rng.integers(0, 4, 3000).astype(np.uint8)
    qry = rng.integers(0, 4, 2000).astype(np.uint8)
    qry[500:1400] = ref[1000:1900]  # one long homology, so some walks reach T
    qry[600:610] = 4
    anchors = np.array([[1000 + i, 500 + i] for i in range(0, 900, 37)]
                       + [[int(rng.integers(0, 3000)), int(rng.integers(0, 2000))] for _ in range(60)]
                       + [[0, 5], [7, 0], [2999, 1999], [2999, 3]], dtype=np.uint32)
    X = 300
    want = 0
    for ar, aq in anchors.astype(np.int64):
        nl, ml = _side_pairs_np(m, ref, qry, ar, aq, False, X, T)
        want += nl
        if ml < T:
            nr, _ = _side_pairs_np(m, ref, qry, ar, aq, True, X, T - ml)
            want += nr
    assert oracle.gate_pairs(ref, qry, anchors, m, X, T) == want


def test_gate_pairs_closed_forms():
    m = hoxd70()
    s = np.full(500, 1, dtype=np.uint8)  # all C: every pair scores 100
    # T out of reach: both walks run to the edges
    assert oracle.gate_pairs(s, s, np.array([[200, 200]], np.uint32), m, 910, 10 ** 9) == 500
    # left maximum reaches T = 1000 after 10 pairs: the right walk is not needed
    assert oracle.gate_pairs(s, s, np.array([[200, 200]], np.uint32), m, 910, 1000) == 10
    # left walk has 4 pairs (400), the right needs 6 more
    assert oracle.gate_pairs(s, s, np.array([[4, 4]], np.uint32), m, 910, 1000) == 4 + 6
    assert oracle.gate_pairs(s, s, np.zeros((0, 2), np.uint32), m, 910, 1000) == 0


# ---------------------------------------------------------------- gate flags (D.2/D.3: flag = total >= T)

def _hand_gate_case():
    """Anchor at 5 of a 10-base pair of sequences under the hand matrix.

    Left side (bases 4, 3, 2, 1, 0, outward): ref C/query A +40, then A/C
    -10, A/A +10, A/A +10, A/C -10: running sums 40, 30, 40, 50, 40, so the
    left maximum is 50 (4 bases).  Right side (bases 5..9): A/A +10, A/C -10,
    A/C -10, G/G +50, T/A -100: sums 10, 0, -10, 40, -60, so the right
    maximum is 40 with X = 20 (deficit exactly X is not a stop) and 10 with
    X = 19 (the walk stops at the third base).  Totals: 90 and 60.
    """
    ref = _seq("AAAAC" + "AAAGT")
    qry = _seq("CAACA" + "ACCGA")
    return ref, qry, np.array([[5, 5]], np.uint32)


def test_gate_flag_at_exactly_T_and_T_minus_1():
    m = _hand_matrix()
    ref, qry, a = _hand_gate_case()
    sc = oracle.side_scores(ref, qry, a, m, 20)[0]
    assert sc.tolist() == [50, 4, 40, 4]
    assert oracle.gate(ref, qry, a, m, 20, 90).tolist() == [1]
    assert oracle.gate(ref, qry, a, m, 20, 91).tolist() == [0]
    # X = 19 stops the right walk before its +50 base: total 60
    assert oracle.gate(ref, qry, a, m, 19, 60).tolist() == [1]
    assert oracle.gate(ref, qry, a, m, 19, 61).tolist() == [0]
    assert oracle.gate(ref, qry, a, m, 19, 90).tolist() == [0]


def test_gate_rejected_slot_of_materialize_is_zero():
    m = _hand_matrix()
    ref, qry, a = _hand_gate_case()
    rec, done = oracle.materialize(ref, qry, a, 0, [0], m, 20, 91)
    assert rec[0].tolist() == [0, 0, 0, 0] and done[0] == 0
    # at T = total the same id is accepted: left extent 4, right extent 4 bases
    rec, done = oracle.materialize(ref, qry, a, 0, [0], m, 20, 90)
    assert rec[0].tolist() == [1, 1, 7, 90] and done[0] == 1
    # ids are global: with id_base 7, id 7 addresses the same anchor 0
    rec, done = oracle.materialize(ref, qry, a, 7, [7], m, 20, 91)
    assert rec[0].tolist() == [0, 0, 0, 0] and done[0] == 0


def _random_gate_case(seed, L=90, n_anchor=60):
    rng = np.random.default_rng(seed)
    ref = rng.integers(0, 5, L).astype(np.uint8)
    qry = np.where(rng.random(L) < 0.55, ref, rng.integers(0, 5, L)).astype(np.uint8)
    m = rng.integers(-60, 61, (5, 5)).astype(np.int32)  # asymmetric
    anchors = np.stack([rng.integers(0, L, n_anchor), rng.integers(0, L, n_anchor)], 1).astype(np.uint32)
    anchors[: n_anchor // 3, 1] = anchors[: n_anchor // 3, 0]  # some on the main diagonal (long walks)
    return ref, qry, m, anchors


@pytest.mark.parametrize("seed", range(6))
def test_gate_at_infinite_x_is_best_window_through_the_anchor(seed):
    """X = infinity: the walk never stops before an edge, so the total is the
    best score of any window [a-l, a+r) around the anchor (the empty window
    scores 0), found here by enumerating every (l, r)."""
    ref, qry, m, anchors = _random_gate_case(seed)
    best = []
    for ar, aq in anchors.astype(np.int64):
        b = 0
        for l in range(min(ar, aq) + 1):
            for r in range(min(ref.size - ar, qry.size - aq) + 1):
                s = sum(int(m[ref[ar + k], qry[aq + k]]) for k in range(-l, r))
                b = max(b, s)
        best.append(b)
    best = np.array(best)
    assert best.min() < np.median(best) < best.max()
    for T in (int(np.median(best)), int(np.median(best)) + 1, int(best.max()), int(best.max()) + 1, 1):
        flags = oracle.gate(ref, qry, anchors, m, 1 << 30, T)
        assert flags.tolist() == (best >= T).astype(np.uint8).tolist()
    assert 0 < oracle.gate(ref, qry, anchors, m, 1 << 30, int(np.median(best))).sum() < len(anchors)


def _side_max_np(m, ref, qry, ar, aq, right, X):
    """The X-drop side maximum from prefix sums: n* = the first step whose
    sum falls more than X below the maximum of the sums before it (the
    empty prefix included); the result is the largest sum before n*."""
    if right:
        k = min(ref.size - ar, qry.size - aq)
        sc = m[ref[ar:ar + k], qry[aq:aq + k]].astype(np.int64)
    else:
        k = min(ar, aq)
        sc = m[ref[ar - k:ar][::-1], qry[aq - k:aq][::-1]].astype(np.int64)
    S = np.concatenate([[0], np.cumsum(sc)])
    before = np.maximum.accumulate(S)[:-1]
    drop = np.flatnonzero(before - S[1:] > X)
    stop = drop[0] + 1 if drop.size else S.size
    return int(S[:stop].max())


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("X", [0, 45, 130])
def test_gate_flags_match_prefix_sum_form(seed, X):
    ref, qry, m, anchors = _random_gate_case(100 + seed, L=200, n_anchor=150)
    tot = np.array([_side_max_np(m, ref, qry, ar, aq, False, X) + _side_max_np(m, ref, qry, ar, aq, True, X)
                    for ar, aq in anchors.astype(np.int64)])
    for T in sorted({1, int(np.median(tot)), int(np.median(tot)) + 1, int(tot.max()), int(tot.max()) + 1}):
        T = max(T, 1)
        flags = oracle.gate(ref, qry, anchors, m, X, T)
        assert flags.tolist() == (tot >= T).astype(np.uint8).tolist()


# ---------------------------------------------------------------- digests (test tool, not the method)

def test_fnv1a64_published_vectors_and_streaming():
    """FNV-1a 64 (Fowler, Noll, Vo): the published digests of "", "a" and
    "foobar"; a digest continued over pieces equals the digest of the whole."""
    assert oracle.fnv1a64(b"") == 0xCBF29CE484222325
    assert oracle.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert oracle.fnv1a64(b"foobar") == 0x85944171F73967E8
    data = np.random.default_rng(3).integers(0, 256, 1000).astype(np.uint8)
    h = oracle.fnv1a64(data[:300])
    assert oracle.fnv1a64(data[300:], h) == oracle.fnv1a64(data)
    assert oracle.fnv1a64(data.view(np.uint32)) == oracle.fnv1a64(data)


def test_segment_digests_equal_whole_chunk_arrays(tmp_path):
    """The per-segment oracle pass used for full-size parity gives, segment by
    segment, the digests of the slices of the whole-chunk oracle arrays."""
    from oracle import digest
    from seed_hits_ungapped_gb300 import synth
    w = synth.make("chunking", scale=0.02)
    res = oracle.run_path(w.ref, w.query, w.matrix, w.xdrop, w.K, max_hits=w.max_hits)
    idx, pos = res["idx"], res["pos"]
    np.save(tmp_path / "ref.npy", w.ref)
    np.save(tmp_path / "idx.npy", idx)
    np.save(tmp_path / "pos.npy", pos)
    np.save(tmp_path / "meta.npy", np.zeros(1))
    np.save(tmp_path / "query0.npy", w.query)
    np.save(tmp_path / "buckets0.npy", res["buckets"])
    np.save(tmp_path / "P0.npy", res["P"])
    assert len(res["chunks"]) > 2
    n_seg = 0
    for c, pc in zip(res["chunks"], res["per_chunk"]):
        hb = int(c[2])
        segs = digest.segments(res["P"], c, 997)
        assert segs[0][0] == c[0] and segs[-1][1] == c[1]
        for s0, s1, h0, h1 in segs:
            got = digest.segment_digests((str(tmp_path), 0, (s0, s1, h0, h1), w.matrix, w.xdrop, res["T"], SPAN))
            a0, a1 = h0 - hb, h1 - hb
            sel = (pc["ids"] >= h0) & (pc["ids"] < h1)
            assert got["n_anchors"] == a1 - a0 and got["n_survivors"] == int(sel.sum())
            assert got["anchors"] == oracle.fnv1a64(pc["anchors"][a0:a1])
            assert got["flags"] == oracle.fnv1a64(pc["flags"][a0:a1])
            assert got["ids"] == oracle.fnv1a64(pc["ids"][sel])
            assert got["records"] == oracle.fnv1a64(pc["rec"][sel])
            assert got["done"] == oracle.fnv1a64(pc["done"][sel])
            n_seg += 1
    assert n_seg > 6
