"""Seeded synthetic workloads (inputs only; none of the method's arithmetic).

The same generator feeds the CUDA library, the CPU oracle, the tests and the
benchmark.  Sequences are uint8 base codes A=0 C=1 G=2 T=3 N=4.

Recipe (numpy ``default_rng`` / PCG64, one seed per workload):
  background  -> i.i.d. bases at the stated composition
  overwrites  -> N runs, repeat-element copies, (CA)n microsatellites, poly-A
  homologies  -> segments copied from uniform reference positions into
                 uniform, non-overlapping query positions; every A/C/G/T base
                 of a copy is substituted with probability d (per segment,
                 d ~ U[lo, hi]) by a uniform one of the other three bases; N is
                 copied unchanged.

Workloads (full size at ``scale=1``; ``scale < 1`` shrinks every length and
count in proportion for oracle-sized parity cases):
  tiny      ref 1 Mbp uniform, query 200 kbp uniform, 100 homologies of
            200-2000 bp at 10%; no hit cap.
  mid       ref 20 Mbp at 41% GC with 1% of bases in N runs of 50-500, query
            5 Mbp of the same composition, 2,000 homologies of 100-5000 bp at
            5-30%.
  dense     ref 10 Mbp uniform with one 300 bp element written at 5,000 places
            (15% substitutions each) and (CA)n runs of 20-200 bp covering 2%;
            query 2 Mbp from the same generator (1,000 element copies, 2% (CA)n)
            plus 500 homologies of 200-2000 bp at 10%.
  workload_a ref 100 Mbp at 41% GC, query 25 Mbp at 41% GC, 10,000 homologies
            of 100-3000 bp at 5-25%; one chunk.  Stands in for the pages'
            frozen workload A (hg38 x mm39 unit 0), which is not available.
  chunking  workload_a plus a 4,000 bp poly-A run written into the reference
            and copied into the query; both query strands (forward and reverse
            complement) as separate batches; hit cap 2^24.  (Scaled cases shrink
            the poly-A run with the lengths and the cap with the anchor count.)

Scoring for every workload: HOXD70 (A/C/G/T block) with N scoring -100 against
anything, X-drop 910, hsp threshold K = 3000.
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np

A, C, G, T, N = 0, 1, 2, 3, 4
SEED_PATTERN = "1110100110010101111"

_HOXD70_ACGT = [
    [91, -114, -31, -123],
    [-114, 100, -125, -31],
    [-31, -125, 100, -114],
    [-123, -31, -114, 91],
]


def hoxd70(n_score: int = -100) -> np.ndarray:
    """5x5 int32 matrix, row = reference base, column = query base."""
    m = np.full((5, 5), n_score, dtype=np.int32)
    m[:4, :4] = np.array(_HOXD70_ACGT, dtype=np.int32)
    return m


@dataclasses.dataclass
class Workload:
    name: str
    ref: np.ndarray
    queries: List[np.ndarray]
    matrix: np.ndarray
    xdrop: int = 910
    K: int = 3000
    max_hits: int = 0  # 0 = no cap
    pattern: str = SEED_PATTERN
    seed: int = 0
    scale: float = 1.0

    @property
    def query(self) -> np.ndarray:
        return self.queries[0]


def _background(rng, n: int, p=(0.25, 0.25, 0.25, 0.25)) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    cut = np.cumsum(np.asarray(p, dtype=np.float64))[:3] * 65536.0
    cut = np.round(cut).astype(np.uint32)
    step = 1 << 24
    for s in range(0, n, step):
        e = min(n, s + step)
        u = rng.integers(0, 65536, e - s, dtype=np.uint32)
        out[s:e] = np.searchsorted(cut, u, side="right").astype(np.uint8)
    return out


def _mutate(rng, seg: np.ndarray, d: float) -> np.ndarray:
    seg = seg.copy()
    hit = (rng.random(seg.size) < d) & (seg < 4)
    k = int(hit.sum())
    if k:
        seg[hit] = ((seg[hit].astype(np.int32) + rng.integers(1, 4, k)) % 4).astype(np.uint8)
    return seg


def _overwrite_runs(rng, seq: np.ndarray, fraction: float, lo: int, hi: int, make):
    """Overwrite random runs (lengths U[lo, hi]) until `fraction` of seq is covered."""
    target = int(round(fraction * seq.size))
    done = 0
    while done < target:
        ln = min(int(rng.integers(lo, hi + 1)), seq.size)
        p = int(rng.integers(0, seq.size - ln + 1))
        seq[p:p + ln] = make(ln)
        done += ln


def _plant(rng, ref, qry, n_seg, lo, hi, dlo, dhi, occupied=None):
    """Copy n_seg reference segments into non-overlapping query places."""
    if occupied is None:
        occupied = np.zeros(qry.size, dtype=bool)
    placed = 0
    tries = 0
    while placed < n_seg and tries < 50 * max(1, n_seg):
        tries += 1
        ln = int(rng.integers(lo, hi + 1))
        if ln > min(ref.size, qry.size):
            continue
        src = int(rng.integers(0, ref.size - ln + 1))
        dst = int(rng.integers(0, qry.size - ln + 1))
        if occupied[dst:dst + ln].any():
            continue
        d = float(rng.uniform(dlo, dhi)) if dhi > dlo else float(dlo)
        qry[dst:dst + ln] = _mutate(rng, ref[src:src + ln], d)
        occupied[dst:dst + ln] = True
        placed += 1
    return occupied


def _ca_run(ln: int) -> np.ndarray:
    out = np.empty(ln, dtype=np.uint8)
    out[0::2] = C
    out[1::2] = A
    return out


def reverse_complement(seq: np.ndarray) -> np.ndarray:
    """Minus-strand batch of a query (input preparation for two-strand runs)."""
    lut = np.array([T, G, C, A, N], dtype=np.uint8)
    return lut[seq[::-1]]


GC41 = (0.295, 0.205, 0.205, 0.295)


def _sz(x, scale):
    return max(1, int(round(x * scale)))


def make(name: str, scale: float = 1.0) -> Workload:
    """Build one named workload (deterministic for a given name and scale)."""
    names = ["tiny", "mid", "dense", "workload_a", "chunking"]
    if name not in names:
        raise ValueError("unknown workload %r (one of %s)" % (name, names))
    i = names.index(name)
    seed = 1 if i == 0 else 1 + i
    rng = np.random.default_rng(seed if scale == 1.0 else [seed, int(round(scale * 1e6))])
    m = hoxd70()
    if name == "tiny":
        ref = _background(rng, _sz(1_000_000, scale))
        qry = _background(rng, _sz(200_000, scale))
        _plant(rng, ref, qry, _sz(100, scale), 200, 2000, 0.10, 0.10)
        return Workload(name, ref, [qry], m, seed=seed, scale=scale)
    if name == "mid":
        ref = _background(rng, _sz(20_000_000, scale), GC41)
        qry = _background(rng, _sz(5_000_000, scale), GC41)
        nrun = lambda ln: np.full(ln, N, dtype=np.uint8)  # noqa: E731
        _overwrite_runs(rng, ref, 0.01, 50, 500, nrun)
        _overwrite_runs(rng, qry, 0.01, 50, 500, nrun)
        _plant(rng, ref, qry, _sz(2000, scale), 100, 5000, 0.05, 0.30)
        return Workload(name, ref, [qry], m, seed=seed, scale=scale)
    if name == "dense":
        ref = _background(rng, _sz(10_000_000, scale))
        qry = _background(rng, _sz(2_000_000, scale))
        element = _background(rng, 300)
        for seq, copies in ((ref, _sz(5000, scale)), (qry, _sz(1000, scale))):
            for _ in range(copies):
                p = int(rng.integers(0, seq.size - 300 + 1))
                seq[p:p + 300] = _mutate(rng, element, 0.15)
            _overwrite_runs(rng, seq, 0.02, 20, 200, _ca_run)
        _plant(rng, ref, qry, _sz(500, scale), 200, 2000, 0.10, 0.10)
        return Workload(name, ref, [qry], m, seed=seed, scale=scale)
    # workload_a / chunking
    ref = _background(rng, _sz(100_000_000, scale), GC41)
    qry = _background(rng, _sz(25_000_000, scale), GC41)
    occ = None
    if name == "chunking":
        ln = 4000 if scale == 1.0 else max(40, int(round(4000 * scale)))
        p = int(rng.integers(0, ref.size - ln + 1))
        ref[p:p + ln] = A
        dst = int(rng.integers(0, qry.size - ln + 1))
        qry[dst:dst + ln] = A
        occ = np.zeros(qry.size, dtype=bool)
        occ[dst:dst + ln] = True
    _plant(rng, ref, qry, _sz(10_000, scale), 100, 3000, 0.05, 0.25, occ)
    if name == "workload_a":
        return Workload(name, ref, [qry], m, seed=seed, scale=scale)
    cap = max(1, int(round((1 << 24) * scale * scale)))  # anchors grow with both lengths
    return Workload(name, ref, [qry, reverse_complement(qry)], m, max_hits=cap, seed=seed, scale=scale)


WORKLOADS = ["tiny", "mid", "dense", "workload_a", "chunking"]
