"""Benchmark: seed hits -> anchors -> score gate -> survivors -> SegmentPairs.

One step = the whole path over one synthetic query batch: hit discovery
(count, prefix, chunk walk), fused expansion + score gate, stable compaction,
materialization and the accepted compaction.  The metric is anchors per
second.  "roofline" reports the dominant kernel (fused expansion + gate)
against the measured HBM copy bandwidth: algorithmic bytes (16 per seed, 13
per anchor, both sequences once) per launch over the launch's CUDA-event
time.  That kernel is bound by integer work, not by HBM, so two models are
reported beside it: "alu_model" (4 int32 operations per base pair the gate
decision scores, pairs per anchor measured by the oracle on the CPU sample,
against 128 int32 lanes per SM per cycle) and, from ncu instruction counts
of the same kernel version, "issue_roofline" (issued lane-instructions
against the SMs' issue rate).
Duplicate removal over each batch's accepted HSPs ("dedup") is timed apart
from the step (--no-dedup skips it).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

With N > 1 the script runs under torchrun, one rank per GPU; every rank runs
its own copy of the workload (weak scaling) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "anchors/sec (hit expansion + score gate, device-timed); HBM GB/s vs GB300 peak"
UNIT = "anchors/s"
L2_FLUSH_BYTES = 512 << 20

WORKLOAD_DESC = {
    "workload_a": "workload_a: ref 100 Mbp + query 25 Mbp at 41% GC, 10,000 planted homologies 100-3000 bp at "
                  "5-25% divergence, 12of19 seed, HOXD70, X-drop 910, K 3000, one chunk",
    "tiny": "tiny: ref 1 Mbp + query 200 kbp uniform, 100 homologies 200-2000 bp at 10%",
    "mid": "mid: ref 20 Mbp + query 5 Mbp at 41% GC with 1% N runs, 2,000 homologies 100-5000 bp at 5-30%",
    "dense": "dense: ref 10 Mbp + query 2 Mbp with a 300 bp repeat (5,000/1,000 copies) and 2% (CA)n",
    "chunking": "chunking: workload_a + 4 kbp poly-A, both strands, MAX_HITS 2^24",
}


def algorithmic_bytes(n_seeds: int, n_anchors: int, ref_len: int, qry_len: int) -> int:
    """Compulsory bytes of the fused expansion + gate: 16 per seed (two index
    reads, the prefix, the bucket start), 13 per anchor (4-byte position read,
    8-byte anchor write, 1-byte flag write), and both sequences once."""
    return 16 * n_seeds + 13 * n_anchors + ref_len + qry_len


def workload_desc(args) -> str:
    d = WORKLOAD_DESC.get(args.workload, args.workload)
    return d if args.scale == 1.0 else "%s, scaled by %g (sizes and counts)" % (d, args.scale)


def measured_sm_max_mhz() -> float:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f).get("sm_max_mhz", 2070.0))
    return 2070.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms from before
    the warm-up on; the summary keeps the samples whose timestamps fall in
    the timed region (`window`, wall-clock seconds)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index: int, path: str | None = None):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        self.window = None
        self.path = path or os.path.join(tempfile.gettempdir(), "hspz_bench_clocks_%d_gpu%d.csv"
                                         % (os.getpid(), gpu_index))

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:  # nvidia-smi prints local time, e.g. 2026/12/02 19:59:03.123
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append((ts, parts[1:]))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        where = "all samples"
        if self.window is not None:
            slack = self.INTERVAL_MS / 1e3
            inside = [r for r in rows if self.window[0] - slack <= r[0] <= self.window[1] + slack]
            if inside:
                rows, where = inside, "timed region"
            else:  # a region shorter than the sampling interval: the nearest sample
                mid = 0.5 * (self.window[0] + self.window[1])
                rows, where = [min(rows, key=lambda r: abs(r[0] - mid))], "nearest to the timed region"
        vals = [r[1] for r in rows]
        sm = [float(v[1]) for v in vals if v[1].replace(".", "").isdigit()]
        mx = [float(v[2]) for v in vals if v[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for v in vals for k in range(4) if v[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(vals), "sampled": where}


def host_info():
    """Host cores (nproc) and CPU model of the machine the CPU figures come from.
    Arm cores name no model in /proc/cpuinfo; their implementer and part
    numbers stand in for it."""
    import platform
    fields = {}
    try:
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    model = fields.get("model name")
    if not model and "cpu part" in fields:
        model = "%s, cpu implementer %s, cpu part %s" % (platform.machine(), fields.get("cpu implementer", "?"),
                                                         fields["cpu part"])
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.machine(), "machine": platform.machine()}


def run_cpu_baseline(w, seconds: float = 12.0):
    """The oracle as it stands, single-threaded, on a bounded sample of the
    same workload: expansion + gate over the seeds of the query's leading
    part (index, counts and prefix are set up untimed)."""
    import oracle
    idx, pos = oracle.build_index(w.ref)
    buckets = oracle.seed_buckets(w.query)
    P, total, rc = oracle.inclusive_prefix(oracle.count_hits(idx, buckets))
    T = oracle.keep_threshold(w.K)
    done_anchors, t_used, s_begin = 0, 0.0, 0
    pairs = pair_anchors = 0
    step_seeds = 200_000
    while t_used < seconds and s_begin < P.size:
        s_end = min(P.size, s_begin + step_seeds)
        hb = int(P[s_begin - 1]) if s_begin else 0
        chunk = np.array([s_begin, s_end, hb, P[s_end - 1]], np.uint32)
        t0 = time.perf_counter()
        a = oracle.expand(idx, pos, buckets, P, chunk)
        oracle.gate(w.ref, w.query, a, w.matrix, w.xdrop, T)
        t_used += time.perf_counter() - t0
        done_anchors += len(a)
        # untimed: the base pairs the gate decision needs, on every 16th anchor
        sub = a[::16]
        pair_anchors += len(sub)
        pairs += oracle.gate_pairs(w.ref, w.query, sub, w.matrix, w.xdrop, T)
        s_begin = s_end
    return {"value": done_anchors / t_used, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "expansion + gate of the first %d seeds (%d anchors) of the %s query, single-threaded C"
                      % (s_begin, done_anchors, w.name), "seconds": round(t_used, 3), "host": host_info(),
            "gate_pairs_per_anchor": pairs / pair_anchors if pair_anchors else None,
            "gate_pairs_sample": "oracle.gate_pairs over every 16th of those anchors (%d)" % pair_anchors}


def reference_arm(args):
    """--impl reference: the oracle, timed on the host cores, on bounded samples."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from seed_hits_ungapped_gb300 import synth
    import oracle
    w = synth.make(args.workload, args.scale)
    idx, pos = oracle.build_index(w.ref)
    buckets = oracle.seed_buckets(w.query)
    P, total, rc = oracle.inclusive_prefix(oracle.count_hits(idx, buckets))
    T = oracle.keep_threshold(w.K)
    sample_seeds = 400_000
    times, anchors = [], 0
    for step in range(args.warmup + args.steps):
        s0 = (step * sample_seeds) % max(1, P.size - sample_seeds)
        s1 = min(P.size, s0 + sample_seeds)
        hb = int(P[s0 - 1]) if s0 else 0
        chunk = np.array([s0, s1, hb, P[s1 - 1]], np.uint32)
        t0 = time.perf_counter()
        a = oracle.expand(idx, pos, buckets, P, chunk)
        f = oracle.gate(w.ref, w.query, a, w.matrix, w.xdrop, T)
        ids = oracle.compact(f, hb)
        oracle.materialize(w.ref, w.query, a, hb, ids, w.matrix, w.xdrop, T)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            anchors += len(a)
    value = anchors / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic", "config": {"workload": workload_desc(args)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "per step: expansion + gate + compaction + materialization of %d "
                                       "consecutive seeds of the %s query (single-threaded C oracle)"
                                       % (sample_seeds, w.name), "host": host_info()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="workload_a")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-dedup", action="store_true")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="size factor of the workload (profiling on smaller cases; 1 = the workload as named)")
    ap.add_argument("--gate", default="fused", choices=["fused", "bucketed"],
                    help="fused expansion + gate (default), or expansion then the reference-bucketed gate (D.5)")
    ap.add_argument("--clocks-csv", default=None,
                    help="where to write the nvidia-smi clock samples (default: a file in the temp directory)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import torch.distributed as dist
    from seed_hits_ungapped_gb300 import hspz, synth
    from seed_hits_ungapped_gb300.engine import HspEngine

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    w = synth.make(args.workload, args.scale)
    lib = hspz.load_library()
    eng = HspEngine(w.ref, w.matrix, w.xdrop, w.K)
    stream = torch.cuda.current_stream()
    d_queries = [torch.from_numpy(q).cuda() for q in w.queries]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    ev_gate = []
    gate_ms_list = []

    def step(timed_gate=False):
        """One pass of the whole path over every query batch of the workload."""
        n_anchors = n_seeds = 0
        for dq in d_queries:
            plan = eng.plan(dq, w.max_hits)
            n_seeds += plan.n_seeds
            for c in range(plan.n_chunks):
                if args.gate == "fused":
                    # one C call per chunk: fused expansion + gate, compaction, materialization,
                    # accepted compaction; the fused kernel's own duration comes back event-timed
                    n, _, _, ms = eng.process_chunk(plan, c, time_gate=timed_gate)
                    if timed_gate:
                        gate_ms_list.append(ms)
                else:
                    hb, he = int(plan.chunks[c, 2]), int(plan.chunks[c, 3])
                    n = he - hb
                    anchors = eng.buffer("anchors", n, torch.int32, 2)
                    flags = eng.buffer("flags", n, torch.uint8)
                    if timed_gate:
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                    hspz.hspz_expand(plan, c, anchors)
                    hspz.hspz_score_gate_bucketed(eng.index, plan, anchors, n, eng.params, flags)
                    if timed_gate:
                        e1.record(stream)
                        ev_gate.append((e0, e1))
                    ids, n_surv = eng._compact(flags, n, hb, "ids")
                    rec = eng.buffer("records", n_surv, torch.int32, 4)
                    done = eng.buffer("done", n_surv, torch.uint8)
                    hspz.hspz_materialize_plan(eng.index, plan, anchors, hb, ids, n_surv, eng.params, rec, done)
                    eng._compact(done, n_surv, 0, "accepted")
                n_anchors += n
            plan.close()
        return n_anchors, n_seeds

    # clock samples run from before the warm-up on (nvidia-smi takes a while
    # to start); the summary keeps those inside the timed region
    with ClockSampler(local, args.clocks_csv) as clocks:
        for _ in range(args.warmup):
            step()
        barrier()

        # timed region: K steps, each bracketed by CUDA events on the launching
        # stream, with an L2 flush between steps outside the events
        step_ms = []
        launches0 = lib.hspz_kernel_launches()
        barrier()
        t_wall0, t_epoch0 = time.perf_counter(), time.time()
        for _ in range(args.steps):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            n_anchors, n_seeds = step(timed_gate=True)
            b.record(stream)
            b.synchronize()
            step_ms.append(a.elapsed_time(b))
        barrier()
        t_wall = time.perf_counter() - t_wall0
        clocks.window = (t_epoch0, time.time())
    launches = lib.hspz_kernel_launches() - launches0
    total_ms = sum(step_ms)
    if world > 1:
        t = torch.tensor([total_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    value = world * n_anchors * args.steps / (total_ms / 1e3)

    # dominant kernel: fused expansion + gate (one launch per chunk), CUDA-event time per launch
    gate_ms = gate_ms_list + [e0.elapsed_time(e1) for e0, e1 in ev_gate]
    n_launch = len(gate_ms)
    step_bytes = algorithmic_bytes(n_seeds, n_anchors, w.ref.size * len(w.queries), sum(q.size for q in w.queries))
    alg_bytes_per_launch = step_bytes * args.steps / n_launch
    achieved = step_bytes * args.steps / (sum(gate_ms) / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    # ncu counters of the same kernel version (null once the CUDA sources change)
    traffic = None
    prof = {}
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        try:
            tr = json.load(open(tp))
            if tr.get("workload") == args.workload and args.scale == 1.0 and tr.get("kernel_rev") == kernel_rev():
                prof = tr
                traffic = tr.get("bytes_per_launch")
        except Exception:
            prof = {}
    # the second roofline: issued instructions against the SMs' issue rate
    # (4 schedulers x 32 lanes per SM per cycle at the maximum SM clock)
    issue = None
    if prof.get("warp_inst_per_launch"):
        wi = float(prof["warp_inst_per_launch"])
        t_launch = sum(gate_ms) / n_launch / 1e3
        sms = torch.cuda.get_device_properties(local).multi_processor_count
        sm_mhz = measured_sm_max_mhz()
        peak_issue = sms * 128 * sm_mhz * 1e6 / 1e12
        achieved_issue = wi * 32 / t_launch / 1e12
        issue = {"bound": "issue", "achieved": achieved_issue, "peak": peak_issue,
                 "unit": "T lane-instructions/s (warp instructions x 32)", "frac": achieved_issue / peak_issue,
                 "warp_inst_per_anchor": wi / (n_anchors * args.steps / n_launch),
                 "active_lane_frac": (float(prof["thread_inst_per_launch"]) / (wi * 32)
                                      if prof.get("thread_inst_per_launch") else None),
                 "peak_basis": "%d SMs x 128 x %.0f MHz" % (sms, sm_mhz),
                 "source": prof.get("source")}

    # duplicate removal over each batch's accepted HSPs, timed apart from the step
    dedup = None
    if not args.no_dedup:
        n_acc_all = n_fin_all = 0
        dd_ms = []
        for it in range(args.warmup + 3):
            tot = 0.0
            n_acc_all = n_fin_all = 0
            for dq in d_queries:
                r = eng.run(dq, max_hits=w.max_hits, dedup=True)  # collects the batch's accepted records
                batch = eng._bufs.get("batch_records")
                if not r.n_accepted:
                    continue
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                ids, k = eng.dedup(batch, r.n_accepted)
                e1.record(stream)
                e1.synchronize()
                tot += e0.elapsed_time(e1)
                n_acc_all += r.n_accepted
                n_fin_all += k
            if it >= args.warmup:
                dd_ms.append(tot)
        med = statistics.median(dd_ms)
        dedup = {"records": n_acc_all, "final": n_fin_all, "ms_per_step": med,
                 "records_per_s": n_acc_all / (med / 1e3) if med > 0 else None,
                 "timing": "CUDA events around hspz_dedup (it reads the kept count back to host)"}

    # end to end through the public API with host buffers: HspEngine.run_stream
    # takes the pinned host batches and hands back each batch's results (records,
    # done flags, accepted ids of every chunk) in host memory; the next batch's
    # upload and the finished chunks' downloads run on their own streams while
    # the compute stream works, so the copies of one batch overlap the next batch
    e2e = None
    if not args.no_e2e:
        # the dedup leg's buffers (on dense, 33 GB of collected records) are not
        # part of this path: hand their memory back before it runs
        eng.release_buffers("batch_records", "final_ids")
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        hspz.hspz_release_cached_memory()
        pinned = [torch.from_numpy(q).pin_memory() for q in w.queries]
        h2d = sum(q.numel() for q in pinned)
        n_e2e = max(3, args.steps)
        for _ in eng.run_stream(pinned * args.warmup, max_hits=w.max_hits):
            pass
        barrier()
        d2h = 0
        t0 = time.perf_counter()
        for res in eng.run_stream(pinned * n_e2e, max_hits=w.max_hits):
            for c in res.per_chunk:
                d2h += c.records.nbytes + c.done.nbytes + c.accepted.nbytes
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        if world > 1:  # the slowest rank's wall time; every rank streamed its own batches
            t = torch.tensor([e2e_s], dtype=torch.float64, device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_s = float(t.item())
        e2e = {"value": world * n_anchors * n_e2e / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h // n_e2e, "ms_per_step": 1e3 * e2e_s / n_e2e,
               "steps": n_e2e, "api": "HspEngine.run_stream (batches pipelined: copies overlap compute)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(w)

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    kernel_name = ("k_expand_gate_w (fused expansion + score gate)" if args.gate == "fused" else
                   "expansion + bucket sort + k_gate_rounds (reference-bucketed gate)")
    hbm = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
           "traffic": traffic, "peak_kind": peak_kind, "kernel": kernel_name,
           "kernel_ms_per_launch": sum(gate_ms) / n_launch,
           "algorithmic_bytes_per_launch": alg_bytes_per_launch}
    # a model of the integer work beside the HBM roofline: the base pairs the
    # gate decision scores (per anchor, from the oracle on the CPU sample) x 4
    # integer operations per pair (pair score, running sum, running maximum,
    # drop test), against 128 int32 lanes per SM per cycle.  The step's
    # PRMT, IDP4A and LOP3 run at 64 lanes per SM per cycle on sm_103a, so
    # this peak is the IADD/IMNMX rate, an upper bound, not the kernel's.
    alu = None
    if cpu and cpu.get("gate_pairs_per_anchor"):
        sms = torch.cuda.get_device_properties(local).multi_processor_count
        sm_mhz = measured_sm_max_mhz()
        ppa = cpu["gate_pairs_per_anchor"]
        pairs_launch = ppa * n_anchors * args.steps / n_launch
        t_launch = sum(gate_ms) / n_launch / 1e3
        a_ops = 4 * pairs_launch / t_launch / 1e12
        p_ops = sms * 128 * sm_mhz * 1e6 / 1e12
        alu = {"model": "4 int32 operations per base pair the gate decision scores",
               "achieved": a_ops, "peak": p_ops, "unit": "T int32 ops/s", "frac": a_ops / p_ops,
               "peak_kind": "derived: %d SMs x 128 int32 lanes (IADD/IMNMX rate) x %.0f MHz" % (sms, sm_mhz),
               "kernel": kernel_name, "kernel_ms_per_launch": sum(gate_ms) / n_launch,
               "ops_per_pair": 4, "gate_pairs_per_anchor": ppa, "gate_pairs_per_launch": pairs_launch,
               "pairs_basis": cpu.get("gate_pairs_sample")}
    # survivor, accepted and chunk counts over every query batch of one step
    results = [eng.run(dq, max_hits=w.max_hits) for dq in d_queries]
    n_surv_step = sum(r.n_survivors for r in results)
    n_acc_step = sum(r.n_accepted for r in results)
    n_chunks_step = sum(len(r.chunks) for r in results)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": workload_desc(args), "anchors_per_step": n_anchors,
                   "seeds_per_step": n_seeds, "survivors": n_surv_step, "accepted": n_acc_step,
                   "chunks": n_chunks_step, "l2": "flushed (512 MiB write) between timed steps",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "expand_gate_anchors_per_s": n_anchors * args.steps / (sum(gate_ms) / 1e3),
        "roofline": hbm,
        "alu_model": alu,
        "issue_roofline": issue,
        "dedup": dedup,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def code_only(src: str) -> str:
    """C/CUDA source without comments and blank space (string literals kept)."""
    import re
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_rev(read=None) -> str:
    """Hash of the code (comments and blank space left out) of the sources
    that define the fused expansion + gate kernel: ties stored ncu counters
    to a kernel version.  `read(name)` may supply a file's text."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "seed_hits_ungapped_gb300", "csrc")
    for f in ("hspz_gate.cu", "hspz_walk.cuh", "hspz_internal.cuh"):
        text = read(f) if read else open(os.path.join(d, f)).read()
        h.update(code_only(text).encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    sys.exit(main())
