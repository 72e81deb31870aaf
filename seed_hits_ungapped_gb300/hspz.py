"""Thin ctypes binding of libhspz (include/hspz.h) with the same names.

Argument marshalling only: every step runs in the CUDA library.  Device
buffers are torch CUDA tensors (torch is used for device memory and streams);
their ``data_ptr()`` goes straight to the C ABI.  There is no CPU fallback: if
the library is missing or a call fails, an exception is raised.

Tensor conventions (torch has no unsigned 32-bit arithmetic, so uint32 data
travels in int32 tensors of the same bits):
  sequences  uint8  (n,)          base codes A0 C1 G2 T3, anything else N
  anchors    int32  (cap, 2)      hspz_anchor {ref_end, query_end}
  flags/done uint8  (n,)
  ids        int32  (cap,)        uint32 global anchor ids
  records    int32  (n, 4)        hspz_segment_pair {ref_start, query_start, len, score}
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libhspz.so")

HSPZ_OK, HSPZ_E_INVAL, HSPZ_E_HIT_OVERFLOW, HSPZ_E_CAPACITY, HSPZ_E_CUDA, HSPZ_E_NOMEM, HSPZ_E_UNSUPPORTED = range(7)
HSPZ_EXPAND_AUTO, HSPZ_EXPAND_SPARSE, HSPZ_EXPAND_DENSE = 0, 1, 2
HSPZ_WALK_FULL = 1
DEFAULT_PATTERN = "1110100110010101111"

# every entry point declared in include/hspz.h
EXPORTS = [
    "hspz_strerror", "hspz_last_error", "hspz_abi_version", "hspz_keep_threshold", "hspz_build_index",
    "hspz_index_free", "hspz_index_info", "hspz_index_tables", "hspz_find_hits", "hspz_plan_free",
    "hspz_plan_info", "hspz_plan_chunks", "hspz_plan_prefix", "hspz_expand", "hspz_expand_gate",
    "hspz_score_gate", "hspz_compact", "hspz_materialize", "hspz_chunk_walk_host", "hspz_kernel_launches",
    "hspz_compact_noalloc", "hspz_compact_noalloc_max_flags", "hspz_score_gate_bucketed", "hspz_process_chunk",
    "hspz_gather_records", "hspz_dedup", "hspz_release_cached_memory", "hspz_materialize_grouped",
    "hspz_score_gate_plan", "hspz_materialize_plan",
]


class HspzError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = "%s failed: %s" % (what, _strerror(status))
        if detail:
            msg += " (%s)" % detail
        super().__init__(msg)


class hspz_chunk(ctypes.Structure):
    _fields_ = [("seed_begin", ctypes.c_uint32), ("seed_end", ctypes.c_uint32),
                ("hit_begin", ctypes.c_uint32), ("hit_end", ctypes.c_uint32)]


class hspz_score_params(ctypes.Structure):
    _fields_ = [("matrix", ctypes.c_int32 * 25), ("xdrop", ctypes.c_int32), ("K", ctypes.c_int32)]


_lib = None


def load_library():
    """Load libhspz.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libhspz.so not built at %s: run __graft_entry__.build() "
                          "(seed_hits_ungapped_gb300._build.build())" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, U64, U32, I32, VP = ctypes.POINTER, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_void_p
    sig = {
        "hspz_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "hspz_last_error": (ctypes.c_char_p, []),
        "hspz_abi_version": (ctypes.c_int, []),
        "hspz_release_cached_memory": (ctypes.c_int, []),
        "hspz_keep_threshold": (ctypes.c_int, [I32, P(I32)]),
        "hspz_build_index": (ctypes.c_int, [VP, U64, ctypes.c_char_p, P(VP), VP]),
        "hspz_index_free": (None, [VP]),
        "hspz_index_info": (ctypes.c_int, [VP, P(U64), P(U32), P(U32)]),
        "hspz_index_tables": (ctypes.c_int, [VP, P(VP), P(VP)]),
        "hspz_find_hits": (ctypes.c_int, [VP, VP, U64, U64, U32, P(VP), P(U64), VP]),
        "hspz_plan_free": (None, [VP]),
        "hspz_plan_info": (ctypes.c_int, [VP, P(U64), P(U64), P(U32), P(U64)]),
        "hspz_plan_chunks": (ctypes.c_int, [VP, P(hspz_chunk), U32, P(U32)]),
        "hspz_plan_prefix": (ctypes.c_int, [VP, P(VP)]),
        "hspz_expand": (ctypes.c_int, [VP, U32, ctypes.c_int, VP, U64, VP]),
        "hspz_expand_gate": (ctypes.c_int, [VP, U32, P(hspz_score_params), VP, VP, U64, VP]),
        "hspz_score_gate": (ctypes.c_int, [VP, U64, VP, U64, VP, U64, P(hspz_score_params), VP, VP]),
        "hspz_score_gate_plan": (ctypes.c_int, [VP, VP, VP, U64, P(hspz_score_params), VP, VP]),
        "hspz_compact": (ctypes.c_int, [VP, U64, U32, VP, U64, P(U64), VP]),
        "hspz_materialize": (ctypes.c_int, [VP, U64, U32, VP, U64, VP, U64, VP, U64, P(hspz_score_params), VP, VP,
                                            VP]),
        "hspz_materialize_plan": (ctypes.c_int, [VP, VP, VP, U64, U32, VP, U64, P(hspz_score_params), VP, VP, VP]),
        "hspz_materialize_grouped": (ctypes.c_int, [VP, VP, VP, U64, U32, VP, U64, P(hspz_score_params), VP, VP, VP]),
        "hspz_chunk_walk_host": (ctypes.c_int, [VP, U64, U64, ctypes.c_int, P(hspz_chunk), U32, P(U32)]),
        "hspz_gather_records": (ctypes.c_int, [VP, VP, U64, VP, VP]),
        "hspz_dedup": (ctypes.c_int, [VP, U64, VP, U64, P(U64), VP]),
        "hspz_kernel_launches": (U64, []),
        "hspz_compact_noalloc": (ctypes.c_int, [VP, U64, U32, VP, U64, P(U64), VP]),
        "hspz_compact_noalloc_max_flags": (U64, []),
        "hspz_score_gate_bucketed": (ctypes.c_int, [VP, VP, VP, U64, P(hspz_score_params), U32, VP, VP]),
        "hspz_process_chunk": (ctypes.c_int, [VP, U32, P(hspz_score_params), VP, VP, U64, VP, VP, VP, VP, U64,
                                              P(U64), P(U64), P(ctypes.c_float), VP]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _strerror(status: int) -> str:
    try:
        return load_library().hspz_strerror(status).decode()
    except Exception:
        return "status %d" % status


def _check(rc: int, what: str):
    if rc != HSPZ_OK:
        detail = load_library().hspz_last_error().decode(errors="replace") if rc in (HSPZ_E_CUDA, HSPZ_E_NOMEM) else ""
        raise HspzError(rc, what, detail)


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dptr(t, dtype=None, what="tensor"):
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (what, dtype, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def score_params(matrix, xdrop: int, K: int) -> hspz_score_params:
    p = hspz_score_params()
    m = np.ascontiguousarray(matrix, dtype=np.int32).reshape(25)
    for i in range(25):
        p.matrix[i] = int(m[i])
    p.xdrop = int(xdrop)
    p.K = int(K)
    return p


def hspz_keep_threshold(K: int) -> int:
    T = ctypes.c_int32(0)
    _check(load_library().hspz_keep_threshold(int(K), ctypes.byref(T)), "hspz_keep_threshold")
    return T.value


class Index:
    """Reference side: k-mer index + packed reference (owned by the library)."""

    def __init__(self, handle, ref_len):
        self.handle = handle
        self.ref_len = ref_len
        n = ctypes.c_uint64(0)
        span = ctypes.c_uint32(0)
        w = ctypes.c_uint32(0)
        _check(load_library().hspz_index_info(handle, ctypes.byref(n), ctypes.byref(span), ctypes.byref(w)),
               "hspz_index_info")
        self.n_positions, self.span, self.weight = n.value, span.value, w.value

    def tables(self):
        """(idx, pos) as int32 CUDA tensors viewing the library's buffers (copied)."""
        import torch
        a = ctypes.c_void_p(0)
        b = ctypes.c_void_p(0)
        _check(load_library().hspz_index_tables(self.handle, ctypes.byref(a), ctypes.byref(b)), "hspz_index_tables")
        idx = _copy_device(a.value, 4 ** self.weight)
        pos = _copy_device(b.value, self.n_positions) if self.n_positions else torch.empty(0, dtype=torch.int32,
                                                                                             device="cuda")
        return idx, pos

    def close(self):
        if self.handle:
            load_library().hspz_index_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DeviceView:
    """View of a library-owned device buffer for torch.as_tensor (copied at once)."""

    def __init__(self, ptr: int, n: int, typestr: str = "<i4"):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False), "version": 2}


def _copy_device(ptr: int, n: int):
    import torch
    return torch.as_tensor(_DeviceView(ptr, n), device="cuda").clone()


def hspz_build_index(d_ref, seed_pattern: str = DEFAULT_PATTERN, stream=None) -> Index:
    import torch
    h = ctypes.c_void_p(0)
    rc = load_library().hspz_build_index(_dptr(d_ref, torch.uint8, "d_ref"), d_ref.numel(),
                                         seed_pattern.encode(), ctypes.byref(h), _stream(stream))
    _check(rc, "hspz_build_index")
    return Index(h, d_ref.numel())


class Plan:
    """One query batch: seeds, counts, prefix, chunks and a packed query."""

    def __init__(self, handle, index: Index, query_len: int):
        self.handle = handle
        self.index = index  # keeps the index alive while the plan is
        self.query_len = query_len
        lib = load_library()
        ns, tot, nmax = ctypes.c_uint64(0), ctypes.c_uint64(0), ctypes.c_uint64(0)
        nc = ctypes.c_uint32(0)
        _check(lib.hspz_plan_info(handle, ctypes.byref(ns), ctypes.byref(tot), ctypes.byref(nc), ctypes.byref(nmax)),
               "hspz_plan_info")
        self.n_seeds, self.total_hits, self.n_chunks, self.max_chunk_hits = ns.value, tot.value, nc.value, nmax.value
        arr = (hspz_chunk * max(1, self.n_chunks))()
        got = ctypes.c_uint32(0)
        _check(lib.hspz_plan_chunks(handle, arr, max(1, self.n_chunks), ctypes.byref(got)), "hspz_plan_chunks")
        self.chunks = np.array([[c.seed_begin, c.seed_end, c.hit_begin, c.hit_end] for c in arr[: got.value]],
                               dtype=np.uint32).reshape(-1, 4)

    def prefix(self):
        """Copy of the inclusive prefix P[n_seeds] as an int32 CUDA tensor (uint32 bits)."""
        import torch
        p = ctypes.c_void_p(0)
        _check(load_library().hspz_plan_prefix(self.handle, ctypes.byref(p)), "hspz_plan_prefix")
        if not self.n_seeds:
            return torch.empty(0, dtype=torch.int32, device="cuda")
        return _copy_device(p.value, self.n_seeds)

    def close(self):
        if self.handle:
            load_library().hspz_plan_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def hspz_find_hits(index: Index, d_query, max_hits: int = 0, walk_full: bool = False, stream=None) -> Plan:
    import torch
    h = ctypes.c_void_p(0)
    total = ctypes.c_uint64(0)
    rc = load_library().hspz_find_hits(index.handle, _dptr(d_query, torch.uint8, "d_query"), d_query.numel(),
                                       int(max_hits), HSPZ_WALK_FULL if walk_full else 0, ctypes.byref(h),
                                       ctypes.byref(total), _stream(stream))
    if rc == HSPZ_E_HIT_OVERFLOW:
        err = HspzError(rc, "hspz_find_hits", "total hits %d" % total.value)
        err.total_hits = total.value
        raise err
    _check(rc, "hspz_find_hits")
    return Plan(h, index, d_query.numel())


def hspz_expand(plan: Plan, chunk: int, d_anchors, mode: int = HSPZ_EXPAND_AUTO, stream=None):
    import torch
    rc = load_library().hspz_expand(plan.handle, int(chunk), int(mode), _dptr(d_anchors, torch.int32, "d_anchors"),
                                    d_anchors.numel() // 2, _stream(stream))
    _check(rc, "hspz_expand")


def hspz_expand_gate(plan: Plan, chunk: int, params: hspz_score_params, d_anchors, d_flags, stream=None):
    import torch
    cap = min(d_anchors.numel() // 2, d_flags.numel())
    rc = load_library().hspz_expand_gate(plan.handle, int(chunk), ctypes.byref(params),
                                         _dptr(d_anchors, torch.int32, "d_anchors"),
                                         _dptr(d_flags, torch.uint8, "d_flags"), cap, _stream(stream))
    _check(rc, "hspz_expand_gate")


def hspz_score_gate(d_anchors, n: int, d_ref, d_query, params: hspz_score_params, d_flags, stream=None):
    """Gate n anchors against raw device sequences (uint8 base codes)."""
    import torch
    if d_anchors.numel() < 2 * n or d_flags.numel() < n:
        raise ValueError("buffers shorter than n")
    rc = load_library().hspz_score_gate(_dptr(d_anchors, torch.int32, "d_anchors"), int(n),
                                        _dptr(d_ref, torch.uint8, "d_ref"), d_ref.numel(),
                                        _dptr(d_query, torch.uint8, "d_query"), d_query.numel(),
                                        ctypes.byref(params), _dptr(d_flags, torch.uint8, "d_flags"), _stream(stream))
    _check(rc, "hspz_score_gate")


def hspz_score_gate_plan(index: Index, plan: Plan, d_anchors, n: int, params: hspz_score_params, d_flags,
                         stream=None):
    """Gate n anchors against the packed sequences of an index and its plan."""
    import torch
    if d_anchors.numel() < 2 * n or d_flags.numel() < n:
        raise ValueError("buffers shorter than n")
    rc = load_library().hspz_score_gate_plan(index.handle, plan.handle, _dptr(d_anchors, torch.int32, "d_anchors"),
                                             int(n), ctypes.byref(params), _dptr(d_flags, torch.uint8, "d_flags"),
                                             _stream(stream))
    _check(rc, "hspz_score_gate_plan")


def hspz_score_gate_bucketed(index: Index, plan: Plan, d_anchors, n: int, params: hspz_score_params, d_flags,
                             n_buckets: int = 0, stream=None):
    """D.5: the flags of hspz_score_gate, gated bucket by bucket of reference window."""
    import torch
    if d_anchors.numel() < 2 * n or d_flags.numel() < n:
        raise ValueError("buffers shorter than n")
    rc = load_library().hspz_score_gate_bucketed(index.handle, plan.handle,
                                                 _dptr(d_anchors, torch.int32, "d_anchors"), int(n),
                                                 ctypes.byref(params), int(n_buckets),
                                                 _dptr(d_flags, torch.uint8, "d_flags"), _stream(stream))
    _check(rc, "hspz_score_gate_bucketed")


def hspz_process_chunk(plan: Plan, chunk: int, params: hspz_score_params, d_anchors, d_flags, d_ids, d_records,
                       d_done, d_accepted, stream=None, time_gate: bool = False):
    """One chunk through expansion + gate, compaction, materialization and the
    accepted compaction, with one host synchronization.  Returns
    (n_survivors, n_accepted, gate_ms or None); raises HspzError with
    .needed = n_survivors when the survivor buffers are too small."""
    import torch
    cap_a = min(d_anchors.numel() // 2, d_flags.numel())
    cap_s = min(d_ids.numel(), d_records.numel() // 4, d_done.numel(), d_accepted.numel())
    ns, na = ctypes.c_uint64(0), ctypes.c_uint64(0)
    ms = ctypes.c_float(0.0)
    rc = load_library().hspz_process_chunk(plan.handle, int(chunk), ctypes.byref(params),
                                           _dptr(d_anchors, torch.int32, "d_anchors"),
                                           _dptr(d_flags, torch.uint8, "d_flags"), cap_a,
                                           _dptr(d_ids, torch.int32, "d_ids"), _dptr(d_records, torch.int32, "d_records"),
                                           _dptr(d_done, torch.uint8, "d_done"),
                                           _dptr(d_accepted, torch.int32, "d_accepted"), cap_s, ctypes.byref(ns),
                                           ctypes.byref(na), ctypes.byref(ms) if time_gate else None, _stream(stream))
    if rc == HSPZ_E_CAPACITY:
        err = HspzError(rc, "hspz_process_chunk", "needs %d survivor slots" % ns.value)
        err.needed = ns.value
        raise err
    _check(rc, "hspz_process_chunk")
    return ns.value, na.value, (ms.value if time_gate else None)


def hspz_compact(d_flags, n: int, id_base: int, d_ids, stream=None) -> int:
    import torch
    if d_flags.numel() < n:
        raise ValueError("flags shorter than n")
    out = ctypes.c_uint64(0)
    rc = load_library().hspz_compact(_dptr(d_flags, torch.uint8, "d_flags"), int(n), int(id_base),
                                     _dptr(d_ids, torch.int32, "d_ids"), d_ids.numel(), ctypes.byref(out),
                                     _stream(stream))
    if rc == HSPZ_E_CAPACITY:
        err = HspzError(rc, "hspz_compact", "needs %d ids" % out.value)
        err.needed = out.value
        raise err
    _check(rc, "hspz_compact")
    return out.value


def hspz_compact_noalloc(d_flags, n: int, id_base: int, d_ids, stream=None) -> int:
    """hspz_compact for callers that cannot allocate device memory: the scratch
    is a fixed array inside the library (at most 2^28 flags per call; calls
    that overlap on the GPU share that array and must be serialized)."""
    import torch
    if d_flags.numel() < n:
        raise ValueError("flags shorter than n")
    out = ctypes.c_uint64(0)
    rc = load_library().hspz_compact_noalloc(_dptr(d_flags, torch.uint8, "d_flags"), int(n), int(id_base),
                                             _dptr(d_ids, torch.int32, "d_ids"), d_ids.numel(), ctypes.byref(out),
                                             _stream(stream))
    if rc == HSPZ_E_CAPACITY:
        err = HspzError(rc, "hspz_compact_noalloc", "needs %d ids" % out.value)
        err.needed = out.value
        raise err
    _check(rc, "hspz_compact_noalloc")
    return out.value


def hspz_materialize(d_anchors, id_base: int, d_ids, n_ids: int, d_ref, d_query, params: hspz_score_params,
                     d_out, d_done, stream=None):
    """Materialize survivors against raw device sequences (uint8 base codes)."""
    import torch
    if d_ids.numel() < n_ids or d_out.numel() < 4 * n_ids or d_done.numel() < n_ids:
        raise ValueError("buffers shorter than n_ids")
    rc = load_library().hspz_materialize(_dptr(d_anchors, torch.int32, "d_anchors"), d_anchors.numel() // 2,
                                         int(id_base), _dptr(d_ids, torch.int32, "d_ids"), int(n_ids),
                                         _dptr(d_ref, torch.uint8, "d_ref"), d_ref.numel(),
                                         _dptr(d_query, torch.uint8, "d_query"), d_query.numel(),
                                         ctypes.byref(params), _dptr(d_out, torch.int32, "d_out"),
                                         _dptr(d_done, torch.uint8, "d_done"), _stream(stream))
    _check(rc, "hspz_materialize")


def hspz_materialize_plan(index: Index, plan: Plan, d_anchors, id_base: int, d_ids, n_ids: int,
                          params: hspz_score_params, d_out, d_done, stream=None, grouped: bool = False):
    """Materialize against the packed sequences of an index and its plan;
    grouped=True calls hspz_materialize_grouped (ids taken in diagonal order)."""
    import torch
    if d_ids.numel() < n_ids or d_out.numel() < 4 * n_ids or d_done.numel() < n_ids:
        raise ValueError("buffers shorter than n_ids")
    lib = load_library()
    fn = lib.hspz_materialize_grouped if grouped else lib.hspz_materialize_plan
    rc = fn(index.handle, plan.handle, _dptr(d_anchors, torch.int32, "d_anchors"),
            d_anchors.numel() // 2, int(id_base), _dptr(d_ids, torch.int32, "d_ids"), int(n_ids),
            ctypes.byref(params), _dptr(d_out, torch.int32, "d_out"),
            _dptr(d_done, torch.uint8, "d_done"), _stream(stream))
    _check(rc, "hspz_materialize_grouped" if grouped else "hspz_materialize_plan")


def hspz_release_cached_memory():
    """Return the library pools' cached device memory to the driver."""
    _check(load_library().hspz_release_cached_memory(), "hspz_release_cached_memory")


def hspz_gather_records(d_records, d_idx, n: int, d_out, stream=None):
    """d_out[k] = d_records[d_idx[k]] for k < n ((m, 4) int32 record tensors)."""
    import torch
    if d_idx.numel() < n or d_out.numel() < 4 * n:
        raise ValueError("buffers shorter than n")
    rc = load_library().hspz_gather_records(_dptr(d_records, torch.int32, "d_records"), _dptr(d_idx, torch.int32, "d_idx"),
                                            int(n), _dptr(d_out, torch.int32, "d_out"), _stream(stream))
    _check(rc, "hspz_gather_records")


def hspz_dedup(d_records, n: int, d_keep_ids, stream=None) -> int:
    """Indices of the first of every group of equal records among the first n,
    in increasing order, into d_keep_ids; returns their count."""
    import torch
    if d_records.numel() < 4 * n:
        raise ValueError("records shorter than n")
    out = ctypes.c_uint64(0)
    rc = load_library().hspz_dedup(_dptr(d_records, torch.int32, "d_records"), int(n),
                                   _dptr(d_keep_ids, torch.int32, "d_keep_ids"), d_keep_ids.numel(),
                                   ctypes.byref(out), _stream(stream))
    if rc == HSPZ_E_CAPACITY:
        err = HspzError(rc, "hspz_dedup", "needs %d ids" % out.value)
        err.needed = out.value
        raise err
    _check(rc, "hspz_dedup")
    return out.value


def hspz_chunk_walk_host(prefix: np.ndarray, max_hits: int, use_block_sums: bool = True) -> np.ndarray:
    P = np.ascontiguousarray(prefix, dtype=np.uint32)
    lib = load_library()
    cap = 64
    while True:
        arr = (hspz_chunk * cap)()
        n = ctypes.c_uint32(0)
        rc = lib.hspz_chunk_walk_host(ctypes.c_void_p(P.ctypes.data if P.size else 0), P.size, int(max_hits),
                                      1 if use_block_sums else 0, arr, cap, ctypes.byref(n))
        if rc == HSPZ_E_CAPACITY:
            cap = n.value
            continue
        _check(rc, "hspz_chunk_walk_host")
        return np.array([[c.seed_begin, c.seed_end, c.hit_begin, c.hit_end] for c in arr[: n.value]],
                        dtype=np.uint32).reshape(-1, 4)
