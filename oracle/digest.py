"""Full-size parity by digest: the oracle's path over one segment of a chunk.

TEST INFRASTRUCTURE (see the package docstring): only ``tests/`` use it.

A segment is a run of whole seeds [s0, s1) inside one MAX_HITS chunk
("C. Hit discovery", C.3); its anchors are the global ids [P[s0-1], P[s1-1]).
``segment_digests`` runs the oracle's steps on it in the pages' order --
backward expansion (C.5), gate (D.2/D.3), stable compaction with global ids
(D.4), materialization of the survivors (E.1-E.5) -- and returns the FNV-1a
64-bit digest of each array plus its length.  Segments are independent, so
a process pool can digest a full-size workload; the arrays are read from
``.npy`` files (memory-mapped) that the caller wrote once.
"""
from __future__ import annotations

import os

import numpy as np

import oracle

_cache = {}


def _arrays(folder: str):
    if folder not in _cache:
        load = lambda name: np.load(os.path.join(folder, name + ".npy"), mmap_mode="r")  # noqa: E731
        meta = np.load(os.path.join(folder, "meta.npy"))
        _cache.clear()
        _cache[folder] = dict(ref=load("ref"), idx=load("idx"), pos=load("pos"), meta=meta,
                              queries={}, load=load)
    return _cache[folder]


def _query(folder: str, strand: int):
    d = _arrays(folder)
    if strand not in d["queries"]:
        d["queries"][strand] = (d["load"]("query%d" % strand), d["load"]("buckets%d" % strand),
                                d["load"]("P%d" % strand))
    return d["queries"][strand]


def segments(P: np.ndarray, chunk, max_anchors: int):
    """Seed-aligned segments of one chunk (seed_begin, seed_end, hit_begin,
    hit_end), each holding at most max_anchors anchors unless one seed alone
    holds more."""
    sb, se, hb, he = (int(x) for x in chunk)
    out = []
    s = sb
    while s < se:
        start = int(P[s - 1]) if s else 0
        # last seed whose inclusive prefix stays within start + max_anchors
        e = int(np.searchsorted(P[s:se], start + max_anchors, side="right")) + s
        e = max(e, s + 1)
        out.append((s, e, start, int(P[e - 1])))
        s = e
    assert out[0][2] == hb and out[-1][3] == he
    return out


def segment_digests(job):
    """job = (folder, strand, (s0, s1, h0, h1), matrix, xdrop, T, span).

    Returns dict(n_anchors, n_survivors, n_accepted, and the FNV-1a 64
    digests of anchors (uint32 pairs), flags (uint8), ids (uint32, global),
    records (int32 x 4) and done flags (uint8))."""
    folder, strand, seg, matrix, xdrop, T, span = job
    d = _arrays(folder)
    qry, buckets, P = _query(folder, strand)
    s0, s1, h0, h1 = seg
    chunk = np.array([s0, s1, h0, h1], np.uint32)
    anchors = oracle.expand(d["idx"], d["pos"], buckets, P, chunk, span)
    flags = oracle.gate(d["ref"], qry, anchors, matrix, xdrop, T)
    ids = oracle.compact(flags, h0)
    rec, done = oracle.materialize(d["ref"], qry, anchors, h0, ids, matrix, xdrop, T)
    return dict(n_anchors=int(anchors.shape[0]), n_survivors=int(ids.size), n_accepted=int(done.sum()),
                anchors=oracle.fnv1a64(anchors), flags=oracle.fnv1a64(flags), ids=oracle.fnv1a64(ids),
                records=oracle.fnv1a64(rec), done=oracle.fnv1a64(done))
