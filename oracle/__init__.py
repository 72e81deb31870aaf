"""Plain CPU oracle for the hspZ seed-hit -> ungapped X-drop HSP path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``seed_hits_ungapped_gb300``) never imports it.

The arithmetic lives in ``hspz_oracle.c`` (plain single-threaded C, written
from the hspZ documentation pages "C. Hit discovery", "D. Score gate" and
"E. X-drop materialization"); this module only marshals numpy arrays through
ctypes.  It shares no code with the CUDA library.

Every function here is pinned in ``tests/test_oracle_pins.py`` against values
fixed by the pages or by the mathematics (worked prefix example, brute-force
seed matching, closed forms, maximum-prefix-sum brute force, tie and drop
boundary hand cases, exhaustive f32 threshold check, the 2^32 refusal edge).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hspz_oracle.c")
_LIB = os.path.join(_HERE, "libhspz_oracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_E_INVAL, ORC_E_OVERFLOW, ORC_E_CAPACITY = 0, 1, 2, 3
SEED_PATTERN = "1110100110010101111"


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: runs on x86-64 and aarch64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            U64 = ctypes.c_uint64
            I32 = ctypes.c_int32
            lib.orc_pattern_info.argtypes = [ctypes.c_char_p, P, P]
            lib.orc_seed_buckets.argtypes = [P, U64, ctypes.c_char_p, P]
            lib.orc_build_index.argtypes = [P, U64, ctypes.c_char_p, P, P, U64, P]
            lib.orc_count_hits.argtypes = [P, P, U64, P]
            lib.orc_count_hits.restype = None
            lib.orc_inclusive_prefix.argtypes = [P, U64, P, P]
            lib.orc_chunk_walk.argtypes = [P, U64, U64, P, U64, P]
            lib.orc_expand.argtypes = [P, P, P, P, P, ctypes.c_int, P]
            lib.orc_expand.restype = None
            lib.orc_gate_pairs.argtypes = [P, U64, P, U64, P, U64, P, ctypes.c_int32, ctypes.c_int32]
            lib.orc_gate_pairs.restype = U64
            lib.orc_anchor_at.argtypes = [P, P, P, P, U64, ctypes.c_int, U64, P]
            lib.orc_side_scores.argtypes = [P, U64, P, U64, P, U64, P, I32, P]
            lib.orc_side_scores.restype = None
            lib.orc_keep_threshold.argtypes = [I32, P]
            lib.orc_gate.argtypes = [P, U64, P, U64, P, U64, P, I32, I32, P]
            lib.orc_gate.restype = None
            lib.orc_compact.argtypes = [P, U64, ctypes.c_uint32, P]
            lib.orc_compact.restype = U64
            lib.orc_materialize.argtypes = [P, U64, P, U64, P, ctypes.c_uint32, P, U64, P, I32, I32, P, P]
            lib.orc_materialize.restype = None
            lib.orc_dedup.argtypes = [P, U64, P]
            lib.orc_dedup.restype = ctypes.c_int
            lib.orc_fnv1a64.argtypes = [U64, P, U64]
            lib.orc_fnv1a64.restype = U64
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a.size else ctypes.c_void_p(0)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def pattern_info(pattern: str = SEED_PATTERN):
    w = ctypes.c_int(0)
    s = ctypes.c_int(0)
    rc = _load().orc_pattern_info(pattern.encode(), ctypes.byref(w), ctypes.byref(s))
    if rc:
        raise OracleError("bad seed pattern %r" % pattern)
    return w.value, s.value


def seed_buckets(seq, pattern: str = SEED_PATTERN) -> np.ndarray:
    """k-mer of every window start (int64, -1 where a care base is N)."""
    seq = _u8(seq)
    _, span = pattern_info(pattern)
    n = max(0, seq.size - span + 1)
    out = np.empty(n, dtype=np.int64)
    rc = _load().orc_seed_buckets(_p(seq), seq.size, pattern.encode(), _p(out))
    if rc:
        raise OracleError("seed_buckets rc=%d" % rc)
    return out


def build_index(ref, pattern: str = SEED_PATTERN):
    """(idx[4^w] inclusive bucket ends, pos[] reference ends grouped by bucket)."""
    ref = _u8(ref)
    w, span = pattern_info(pattern)
    idx = np.empty(4 ** w, dtype=np.uint32)
    cap = max(0, ref.size - span + 1)
    pos = np.empty(cap, dtype=np.uint32)
    n = ctypes.c_uint64(0)
    rc = _load().orc_build_index(_p(ref), ref.size, pattern.encode(), _p(idx), _p(pos), cap, ctypes.byref(n))
    if rc:
        raise OracleError("build_index rc=%d" % rc)
    return idx, pos[: n.value].copy()


def count_hits(idx: np.ndarray, buckets: np.ndarray) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    buckets = np.ascontiguousarray(buckets, dtype=np.int64)
    cnt = np.empty(buckets.size, dtype=np.uint32)
    _load().orc_count_hits(_p(idx), _p(buckets), buckets.size, _p(cnt))
    return cnt


def inclusive_prefix(cnt: np.ndarray):
    """(P, total, rc) -- rc == ORC_E_OVERFLOW when total > 2^32 - 1."""
    cnt = np.ascontiguousarray(cnt, dtype=np.uint32)
    P = np.empty(cnt.size, dtype=np.uint32)
    total = ctypes.c_uint64(0)
    rc = _load().orc_inclusive_prefix(_p(cnt), cnt.size, _p(P), ctypes.byref(total))
    return P, total.value, rc


def chunk_walk(P: np.ndarray, max_hits: int) -> np.ndarray:
    """(n_chunks, 4) uint32: seed_begin, seed_end, hit_begin, hit_end."""
    P = np.ascontiguousarray(P, dtype=np.uint32)
    cap = 16
    while True:
        out = np.empty((cap, 4), dtype=np.uint32)
        n = ctypes.c_uint64(0)
        rc = _load().orc_chunk_walk(_p(P), P.size, int(max_hits), _p(out), cap, ctypes.byref(n))
        if rc == ORC_E_CAPACITY:
            cap *= 4
            continue
        if rc:
            raise OracleError("chunk_walk rc=%d" % rc)
        return out[: n.value].copy()


def expand(idx, pos, buckets, P, chunk, span: int = 19) -> np.ndarray:
    """Anchors of one chunk: (hits, 2) uint32 of (ref_end, query_end)."""
    chunk = np.ascontiguousarray(chunk, dtype=np.uint32).reshape(4)
    n = int(chunk[3]) - int(chunk[2])
    out = np.empty((n, 2), dtype=np.uint32)
    if n:
        _load().orc_expand(_p(np.ascontiguousarray(idx, dtype=np.uint32)),
                           _p(np.ascontiguousarray(pos, dtype=np.uint32)),
                           _p(np.ascontiguousarray(buckets, dtype=np.int64)),
                           _p(np.ascontiguousarray(P, dtype=np.uint32)), _p(chunk), span, _p(out))
    return out


def anchors_at(idx, pos, buckets, P, ids, span: int = 19) -> np.ndarray:
    """Anchors of the given global ids, computed one by one."""
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    pos = np.ascontiguousarray(pos, dtype=np.uint32)
    buckets = np.ascontiguousarray(buckets, dtype=np.int64)
    P = np.ascontiguousarray(P, dtype=np.uint32)
    lib = _load()
    out = np.empty((len(ids), 2), dtype=np.uint32)
    one = np.empty(2, dtype=np.uint32)
    for k, g in enumerate(ids):
        rc = lib.orc_anchor_at(_p(idx), _p(pos), _p(buckets), _p(P), P.size, span, int(g), _p(one))
        if rc:
            raise OracleError("anchor id %d out of range" % g)
        out[k] = one
    return out


def _mat(matrix) -> np.ndarray:
    m = np.ascontiguousarray(matrix, dtype=np.int32).reshape(25)
    return m


def side_scores(ref, qry, anchors, matrix, xdrop: int) -> np.ndarray:
    """(n, 4) int64: M_left, n_left, M_right, n_right per anchor."""
    ref, qry = _u8(ref), _u8(qry)
    a = np.ascontiguousarray(anchors, dtype=np.uint32).reshape(-1, 2)
    out = np.empty((a.shape[0], 4), dtype=np.int64)
    if a.shape[0]:
        _load().orc_side_scores(_p(ref), ref.size, _p(qry), qry.size, _p(a), a.shape[0],
                                _p(_mat(matrix)), int(xdrop), _p(out))
    return out


def keep_threshold(K: int) -> int:
    T = ctypes.c_int32(0)
    rc = _load().orc_keep_threshold(int(K), ctypes.byref(T))
    if rc:
        raise OracleError("keep_threshold: K must be >= 1")
    return T.value


def gate(ref, qry, anchors, matrix, xdrop: int, T: int) -> np.ndarray:
    ref, qry = _u8(ref), _u8(qry)
    a = np.ascontiguousarray(anchors, dtype=np.uint32).reshape(-1, 2)
    flags = np.empty(a.shape[0], dtype=np.uint8)
    if a.shape[0]:
        _load().orc_gate(_p(ref), ref.size, _p(qry), qry.size, _p(a), a.shape[0],
                         _p(_mat(matrix)), int(xdrop), int(T), _p(flags))
    return flags


def gate_pairs(ref, qry, anchors, matrix, xdrop: int, T: int) -> int:
    """Base pairs the gate decision of these anchors scores (a measure of its
    work): each left walk up to its stop, edge or maximum >= T, then, unless
    it reached T, the right walk up to its stop, edge or left + right
    maximum >= T."""
    ref, qry = _u8(ref), _u8(qry)
    a = np.ascontiguousarray(anchors, dtype=np.uint32).reshape(-1, 2)
    if not a.shape[0]:
        return 0
    return int(_load().orc_gate_pairs(_p(ref), ref.size, _p(qry), qry.size, _p(a), a.shape[0],
                                      _p(_mat(matrix)), int(xdrop), int(T)))


def compact(flags, id_base: int = 0) -> np.ndarray:
    flags = _u8(flags)
    ids = np.empty(flags.size, dtype=np.uint32)
    k = _load().orc_compact(_p(flags), flags.size, int(id_base), _p(ids)) if flags.size else 0
    return ids[:k].copy()


def materialize(ref, qry, anchors, id_base: int, ids, matrix, xdrop: int, T: int):
    """(records (n,4) int32 [ref_start, query_start, len, score], done (n,) uint8)."""
    ref, qry = _u8(ref), _u8(qry)
    a = np.ascontiguousarray(anchors, dtype=np.uint32).reshape(-1, 2)
    ids = np.ascontiguousarray(ids, dtype=np.uint32)
    rec = np.empty((ids.size, 4), dtype=np.int32)
    done = np.empty(ids.size, dtype=np.uint8)
    if ids.size:
        _load().orc_materialize(_p(ref), ref.size, _p(qry), qry.size, _p(a), int(id_base), _p(ids), ids.size,
                                _p(_mat(matrix)), int(xdrop), int(T), _p(rec), _p(done))
    return rec, done


def dedup(records):
    """keep (n,) uint8: 1 for the first record, in the given order, of every
    group of records equal in all four fields (see orc_dedup)."""
    rec = np.ascontiguousarray(records, dtype=np.int32).reshape(-1, 4)
    keep = np.zeros(rec.shape[0], dtype=np.uint8)
    if rec.shape[0]:
        rc = _load().orc_dedup(_p(rec), rec.shape[0], _p(keep))
        if rc:
            raise OracleError("orc_dedup failed (%d)" % rc)
    return keep


def run_path(ref, qry, matrix, xdrop: int, K: int, max_hits: int = 0, pattern: str = SEED_PATTERN,
             index=None):
    """The whole path for one query batch, step by step (small inputs only).

    Returns a dict with buckets, counts, P, total, rc, chunks and, per chunk,
    anchors, flags, survivor ids, records and done flags; then the accepted
    records of the batch in raw order ("accepted_rec") and the ones kept by
    dedup ("final_idx" into accepted_rec, "final_rec").
    """
    _, span = pattern_info(pattern)
    idx, pos = index if index is not None else build_index(ref, pattern)
    buckets = seed_buckets(qry, pattern)
    cnt = count_hits(idx, buckets)
    P, total, rc = inclusive_prefix(cnt)
    res = dict(idx=idx, pos=pos, buckets=buckets, cnt=cnt, P=P, total=total, rc=rc, chunks=None, per_chunk=[])
    if rc:
        return res
    T = keep_threshold(K)
    res["T"] = T
    chunks = chunk_walk(P, max_hits)
    res["chunks"] = chunks
    for c in chunks:
        anchors = expand(idx, pos, buckets, P, c, span)
        flags = gate(ref, qry, anchors, matrix, xdrop, T)
        ids = compact(flags, int(c[2]))
        rec, done = materialize(ref, qry, anchors, int(c[2]), ids, matrix, xdrop, T)
        acc = compact(done, 0)
        res["per_chunk"].append(dict(anchors=anchors, flags=flags, ids=ids, rec=rec, done=done, accepted=acc))
    parts = [pc["rec"][pc["accepted"]] for pc in res["per_chunk"]]
    accepted_rec = np.concatenate(parts) if parts else np.zeros((0, 4), np.int32)
    keep = dedup(accepted_rec)
    res["accepted_rec"] = accepted_rec
    res["final_idx"] = np.flatnonzero(keep).astype(np.uint32)
    res["final_rec"] = accepted_rec[keep.astype(bool)]
    return res


FNV64_OFFSET = 14695981039346656037


def fnv1a64(data, h: int = FNV64_OFFSET) -> int:
    """FNV-1a 64-bit digest of an array's bytes (or bytes), continuing from h.
    A test tool, not part of the method (see orc_fnv1a64)."""
    a = np.ascontiguousarray(np.frombuffer(data, np.uint8) if isinstance(data, (bytes, bytearray)) else data)
    b = a.reshape(-1).view(np.uint8)
    return int(_load().orc_fnv1a64(int(h), _p(b), b.size))
