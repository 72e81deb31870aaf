"""One query batch through the whole path, as a sequence of C-ABI calls.

``HspEngine`` owns a reference index and reusable device buffers; ``run``
takes one query batch (a CUDA uint8 tensor) and, per MAX_HITS chunk, calls
hspz_expand_gate -> hspz_compact -> hspz_materialize -> hspz_compact (accepted);
``run_stream`` takes batches in host memory and overlaps their copies with
the compute of neighbouring batches.
Every step runs in libhspz; this module only allocates torch buffers and
passes pointers.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

from . import hspz


@dataclasses.dataclass
class ChunkResult:
    hit_begin: int
    n_anchors: int
    n_survivors: int
    n_accepted: int
    anchors: Optional[np.ndarray] = None   # (n, 2) uint32, when kept
    flags: Optional[np.ndarray] = None     # (n,) uint8
    ids: Optional[np.ndarray] = None       # (n_survivors,) uint32 global anchor ids
    records: Optional[np.ndarray] = None   # (n_survivors, 4) int32 SegmentPairs
    done: Optional[np.ndarray] = None      # (n_survivors,) uint8
    accepted: Optional[np.ndarray] = None  # (n_accepted,) uint32 indices into the survivor list


@dataclasses.dataclass
class BatchResult:
    n_seeds: int
    total_hits: int
    chunks: np.ndarray
    per_chunk: List[ChunkResult]
    prefix: Optional[np.ndarray] = None
    # with dedup: the final HSPs, i.e. the batch's accepted records in raw
    # order with exact duplicates dropped (first kept)
    n_final: int = 0
    d_final: Optional[object] = None                # (n_final, 4) int32 device tensor
    final_records: Optional[np.ndarray] = None      # host copy, with keep or fetch
    final_idx: Optional[np.ndarray] = None          # kept indices into the accepted list, with keep

    @property
    def n_survivors(self):
        return sum(c.n_survivors for c in self.per_chunk)

    @property
    def n_accepted(self):
        return sum(c.n_accepted for c in self.per_chunk)


def _np_u32(t):
    return t.cpu().numpy().view(np.uint32)


class HspEngine:
    """Reference index + scoring parameters + device buffers for repeated batches."""

    def __init__(self, ref, matrix, xdrop: int, K: int, pattern: str = hspz.DEFAULT_PATTERN, stream=None,
                 group: bool = False):
        import torch
        self.torch = torch
        if not torch.cuda.is_available():
            raise RuntimeError("HspEngine needs a CUDA device (the path has no CPU implementation)")
        d_ref = ref if isinstance(ref, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(ref, np.uint8))
        d_ref = d_ref.to(device="cuda", dtype=torch.uint8).contiguous()
        self.stream = stream
        self.group = group  # materialize repetitive chunks in diagonal order
        self.index = hspz.hspz_build_index(d_ref, pattern, stream=stream)
        self.ref_len = d_ref.numel()
        self.params = hspz.score_params(matrix, xdrop, K)
        self.T = hspz.hspz_keep_threshold(K)
        self._bufs = {}
        self._host_bufs = {}

    def buffer(self, name: str, n: int, dtype, cols: int = 1):
        """A reusable device buffer with room for n rows (grown geometrically)."""
        torch = self.torch
        have = self._bufs.get(name)
        if have is None or have.shape[0] < n:
            rows = max(n, int(1.25 * have.shape[0]) if have is not None else n, 1)
            shape = (rows, cols) if cols > 1 else (rows,)
            if have is not None:
                del self._bufs[name]
                del have
            self._bufs[name] = torch.empty(shape, dtype=dtype, device="cuda")
        return self._bufs[name]

    def _compact(self, flags, n, id_base, name):
        torch = self.torch
        ids = self.buffer(name, max(1, n // 64), torch.int32)
        try:
            return ids, hspz.hspz_compact(flags, n, id_base, ids, stream=self.stream)
        except hspz.HspzError as e:
            if e.status != hspz.HSPZ_E_CAPACITY:
                raise
            ids = self.buffer(name, e.needed, torch.int32)
            return ids, hspz.hspz_compact(flags, n, id_base, ids, stream=self.stream)

    def _process_chunk_grouped(self, plan, c: int, n: int, anchors, flags, bufset: str, time_gate: bool = False):
        """A repetitive chunk step by step: fused expansion + gate, compaction,
        materialization in diagonal order, accepted compaction (two host
        synchronizations instead of one).  time_gate: the fused launch's
        duration from events on the engine's stream."""
        torch = self.torch
        hb = int(plan.chunks[c, 2])
        ks = self._torch_stream()
        if time_gate:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(ks)
        hspz.hspz_expand_gate(plan, c, self.params, anchors, flags, stream=self.stream)
        if time_gate:
            e1.record(ks)
        ids, ns = self._compact(flags, n, hb, "ids" + bufset)
        rec = self.buffer("records" + bufset, max(ns, 1), torch.int32, 4)
        done = self.buffer("done" + bufset, max(ns, 1), torch.uint8)
        if ns:
            hspz.hspz_materialize_plan(self.index, plan, anchors, hb, ids, ns, self.params, rec, done,
                                  stream=self.stream, grouped=True)
        acc = self.buffer("accepted" + bufset, max(ns, 1), torch.int32)
        na = hspz.hspz_compact(done, ns, 0, acc, stream=self.stream) if ns else 0
        return n, ns, na, (e0.elapsed_time(e1) if time_gate else None)

    def _torch_stream(self):
        torch = self.torch
        if self.stream is None:
            return torch.cuda.current_stream()
        if isinstance(self.stream, int):
            return torch.cuda.ExternalStream(self.stream)
        return self.stream

    def _host_rows(self, name: str, k: int, n: int, dtype, cols: int = 1, stream=None):
        """Room for n more rows after the first k of a pinned host buffer
        (grown geometrically; the first k rows are kept).  `stream`: the
        stream whose copies may still land in it (default: the engine's)."""
        torch = self.torch
        have = self._host_bufs.get(name)
        if have is None or have.shape[0] < k + n:
            rows = max(k + n, int(1.5 * have.shape[0]) if have is not None else 0, 1024)
            new = torch.empty((rows, cols) if cols > 1 else (rows,), dtype=dtype, pin_memory=True)
            if have is not None and k:
                (stream or self._torch_stream()).synchronize()  # copies still landing in the old buffer
                new[:k].copy_(have[:k])
            self._host_bufs[name] = new
        return self._host_bufs[name]

    def _append_rows(self, name: str, k: int, n: int, cols: int):
        """Room for n more rows after the first k of an int32 buffer, keeping them."""
        torch = self.torch
        have = self._bufs.get(name)
        if have is None or have.shape[0] < k + n:
            rows = max(k + n, int(1.25 * have.shape[0]) if have is not None else 0, 1024)
            new = torch.empty((rows, cols), dtype=torch.int32, device="cuda")
            if have is not None and k:
                new[:k].copy_(have[:k])
            self._bufs[name] = new
        return self._bufs[name]

    def release_buffers(self, *names):
        """Drops the engine's named device buffers (every one when no name is
        given); their memory goes back to PyTorch's caching allocator."""
        for k in (names or tuple(self._bufs)):
            self._bufs.pop(k, None)

    def dedup(self, d_records, n: int):
        """hspz_dedup into the engine's id buffer: (kept ids tensor, count)."""
        torch = self.torch
        ids = self.buffer("final_ids", max(1, n // 2), torch.int32)
        try:
            return ids, hspz.hspz_dedup(d_records, n, ids, stream=self.stream)
        except hspz.HspzError as e:
            if e.status != hspz.HSPZ_E_CAPACITY:
                raise
            ids = self.buffer("final_ids", e.needed, torch.int32)
            return ids, hspz.hspz_dedup(d_records, n, ids, stream=self.stream)

    def plan(self, d_query, max_hits: int = 0, walk_full: bool = False):
        return hspz.hspz_find_hits(self.index, d_query, max_hits, walk_full, stream=self.stream)

    # with group=True a chunk with at least this many hits per seed is taken as
    # repetitive: the ids of one seed then lie on many diagonals, and
    # materialization in diagonal order (hspz_materialize_grouped) lets the
    # survivors of each diagonal share walks.  It pays when repeats are long
    # (a 4 kbp poly-A run: the chunking workload's step 35.7 -> 27.6 ms with
    # every chunk grouped) and costs more than it saves when they are short
    # ((CA)n runs of 20-200 bp: dense's step 283 -> 506 ms), so it is off by
    # default.
    GROUP_HITS_PER_SEED = 64

    def chunk_is_repetitive(self, plan, c: int) -> bool:
        seeds = int(plan.chunks[c, 1]) - int(plan.chunks[c, 0])
        hits = int(plan.chunks[c, 3]) - int(plan.chunks[c, 2])
        return self.group and seeds > 0 and hits >= self.GROUP_HITS_PER_SEED * seeds

    def process_chunk(self, plan, c: int, time_gate: bool = False, bufset: str = ""):
        """hspz_process_chunk on the engine's buffers, growing the survivor
        buffers and running the chunk again when they are too small.
        `bufset` names a separate set of survivor / result buffers.
        Returns (n_anchors, n_survivors, n_accepted, gate_ms)."""
        torch = self.torch
        n = int(plan.chunks[c, 3]) - int(plan.chunks[c, 2])
        anchors = self.buffer("anchors", n, torch.int32, 2)
        flags = self.buffer("flags", n, torch.uint8)
        ids_name = "ids" + bufset
        if self.chunk_is_repetitive(plan, c):
            return self._process_chunk_grouped(plan, c, n, anchors, flags, bufset, time_gate)
        cap = self._bufs[ids_name].shape[0] if ids_name in self._bufs else max(1024, n // 32)
        while True:
            bufs = [self.buffer(ids_name, cap, torch.int32), self.buffer("records" + bufset, cap, torch.int32, 4),
                    self.buffer("done" + bufset, cap, torch.uint8), self.buffer("accepted" + bufset, cap, torch.int32)]
            try:
                ns, na, ms = hspz.hspz_process_chunk(plan, c, self.params, anchors, flags, *bufs,
                                                     stream=self.stream, time_gate=time_gate)
                return n, ns, na, ms
            except hspz.HspzError as e:
                if e.status != hspz.HSPZ_E_CAPACITY:
                    raise
                cap = int(e.needed * 1.1) + 1024

    def run(self, d_query, max_hits: int = 0, walk_full: bool = False, keep: bool = False,
            fetch: bool = False, dedup: bool = False) -> BatchResult:
        """The whole path over one query batch.  keep=True copies every
        intermediate of every chunk to host (fresh arrays); fetch=True copies
        only the results (records, done flags, accepted ids) of every chunk,
        asynchronously into engine-owned pinned host buffers, and returns
        numpy views of them that stay valid until the engine's next run.
        dedup=True also collects the accepted records of all chunks in raw
        order and drops exact duplicates (hspz_gather_records, hspz_dedup)."""
        torch = self.torch
        plan = self.plan(d_query, max_hits, walk_full)
        out = []
        n_acc_total = 0
        off_s = off_a = 0  # rows of the pinned result buffers used so far
        views = []
        for c in range(plan.n_chunks):
            hb = int(plan.chunks[c, 2])
            n, n_surv, n_acc, _ = self.process_chunk(plan, c)
            anchors, flags = self._bufs["anchors"], self._bufs["flags"]
            ids, rec, done, acc = (self._bufs[k] for k in ("ids", "records", "done", "accepted"))
            r = ChunkResult(hb, n, n_surv, n_acc)
            if keep:
                r.anchors = _np_u32(anchors[:n]).reshape(-1, 2).copy()
                r.flags = flags[:n].cpu().numpy().copy()
                r.ids = _np_u32(ids[:n_surv]).copy()
                r.records = rec[:n_surv].cpu().numpy().copy()
                r.done = done[:n_surv].cpu().numpy().copy()
                r.accepted = _np_u32(acc[:n_acc]).copy()
            elif fetch:
                h_rec = self._host_rows("records", off_s, n_surv, torch.int32, 4)
                h_done = self._host_rows("done", off_s, n_surv, torch.uint8)
                h_acc = self._host_rows("accepted", off_a, n_acc, torch.int32)
                with torch.cuda.stream(self._torch_stream()):
                    h_rec[off_s:off_s + n_surv].copy_(rec[:n_surv], non_blocking=True)
                    h_done[off_s:off_s + n_surv].copy_(done[:n_surv], non_blocking=True)
                    h_acc[off_a:off_a + n_acc].copy_(acc[:n_acc], non_blocking=True)
                views.append((r, off_s, n_surv, off_a, n_acc))
                off_s += n_surv
                off_a += n_acc
            if dedup and n_acc:
                batch = self._append_rows("batch_records", n_acc_total, n_acc, 4)
                hspz.hspz_gather_records(rec, acc, n_acc, batch[n_acc_total:], stream=self.stream)
                n_acc_total += n_acc
            out.append(r)
        if views:
            self._torch_stream().synchronize()
            h_rec, h_done, h_acc = (self._host_bufs[k] for k in ("records", "done", "accepted"))
            for r, os_, ns_, oa, na in views:
                r.records = h_rec[os_:os_ + ns_].numpy()
                r.done = h_done[os_:os_ + ns_].numpy()
                r.accepted = h_acc[oa:oa + na].numpy().view(np.uint32)
        res = BatchResult(plan.n_seeds, plan.total_hits, plan.chunks.copy(), out)
        if keep:
            res.prefix = _np_u32(plan.prefix())
        if dedup:
            batch = self._append_rows("batch_records", n_acc_total, 0, 4)
            ids, n_final = self.dedup(batch, n_acc_total)
            final = self.buffer("final_records", max(1, n_final), torch.int32, 4)
            hspz.hspz_gather_records(batch, ids, n_final, final, stream=self.stream)
            res.n_final = n_final
            res.d_final = final[:n_final]
            if keep or fetch:
                res.final_records = final[:n_final].cpu().numpy()
            if keep:
                res.final_idx = _np_u32(ids[:n_final]).copy()
        plan.close()
        return res

    def run_stream(self, host_queries, max_hits: int = 0):
        """Query batches from host memory through the whole path, pipelined.

        `host_queries` is an iterable of uint8 CPU tensors (pinned, for the
        copies to overlap).  While the compute stream works on batch i, an
        upload stream brings batch i+1 to the device and a copy stream takes
        each finished chunk's results (records, done flags, accepted ids)
        back to pinned host buffers.  Yields one BatchResult per batch, in order, once its
        results are on the host; its arrays stay valid until the generator is
        resumed.  Device query and result buffers alternate between two sets,
        so a set is reused only after its copies have finished (events on the
        streams)."""
        torch = self.torch
        ks = self._torch_stream()
        cs = getattr(self, "_copy_stream", None)
        if cs is None:
            cs = self._copy_stream = torch.cuda.Stream()
        # uploads get a stream of their own: behind a batch's downloads (43 GB
        # on dense) the next batch's upload, and so its plan, would wait
        us = getattr(self, "_upload_stream", None)
        if us is None:
            us = self._upload_stream = torch.cuda.Stream()
        dq = [None, None]
        ev_in = [None, None]

        def upload(q, p):
            n = q.numel()
            have = dq[p]
            if have is None or have.numel() < n:
                dq[p] = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
            with torch.cuda.stream(us):
                dq[p][:n].copy_(q, non_blocking=True)
                ev_in[p] = torch.cuda.Event()
                ev_in[p].record(us)
            return n

        it = iter(host_queries)
        q = next(it, None)
        if q is None:
            return
        n_cur = upload(q, 0)
        ev_out = [None, None]  # per result set: the copies of the last chunk that used it
        n_chunk = 0
        pending = None
        i = 0
        while q is not None:
            p = i & 1
            ks.wait_event(ev_in[p])
            plan = self.plan(dq[p][:n_cur], max_hits)  # reads the query, then the host waits for it
            dq[p].record_stream(ks)
            q = next(it, None)
            n_next = upload(q, 1 - p) if q is not None else 0  # the other buffer's batch is planned
            out, views, off_s, off_a = [], [], 0, 0
            for c in range(plan.n_chunks):
                r_set = n_chunk & 1
                if ev_out[r_set] is not None:
                    ks.wait_event(ev_out[r_set])
                n, n_surv, n_acc, _ = self.process_chunk(plan, c, bufset="_s%d" % r_set)
                r = ChunkResult(int(plan.chunks[c, 2]), n, n_surv, n_acc)
                rec, done, acc = (self._bufs[k + "_s%d" % r_set] for k in ("records", "done", "accepted"))
                h_rec = self._host_rows("records_h%d" % p, off_s, n_surv, torch.int32, 4, stream=cs)
                h_done = self._host_rows("done_h%d" % p, off_s, n_surv, torch.uint8, stream=cs)
                h_acc = self._host_rows("accepted_h%d" % p, off_a, n_acc, torch.int32, stream=cs)
                ev_k = torch.cuda.Event()
                ev_k.record(ks)
                cs.wait_event(ev_k)
                with torch.cuda.stream(cs):
                    h_rec[off_s:off_s + n_surv].copy_(rec[:n_surv], non_blocking=True)
                    h_done[off_s:off_s + n_surv].copy_(done[:n_surv], non_blocking=True)
                    h_acc[off_a:off_a + n_acc].copy_(acc[:n_acc], non_blocking=True)
                    ev_out[r_set] = torch.cuda.Event()
                    ev_out[r_set].record(cs)
                for t in (rec, done, acc):
                    t.record_stream(cs)
                views.append((r, off_s, n_surv, off_a, n_acc))
                out.append(r)
                off_s += n_surv
                off_a += n_acc
                n_chunk += 1
            res = BatchResult(plan.n_seeds, plan.total_hits, plan.chunks.copy(), out)
            plan.close()
            last = torch.cuda.Event()
            last.record(cs)
            if pending is not None:
                yield self._finish_stream(*pending)
            pending = (res, views, last, p)
            n_cur = n_next
            i += 1
        yield self._finish_stream(*pending)

    def _finish_stream(self, res, views, ev, p):
        """Waits for a streamed batch's result copies and attaches host views."""
        ev.synchronize()
        h_rec, h_done, h_acc = (self._host_bufs[k + "_h%d" % p] for k in ("records", "done", "accepted"))
        for r, os_, ns_, oa, na in views:
            r.records = h_rec[os_:os_ + ns_].numpy()
            r.done = h_done[os_:os_ + ns_].numpy()
            r.accepted = h_acc[oa:oa + na].numpy().view(np.uint32)
        return res
