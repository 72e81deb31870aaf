"""Host-side parts of the benchmark, no GPU: the algorithmic byte count and
the CPU leg (the oracle's expansion + gate on a bounded sample, and the base
pairs per anchor that the ALU roofline counts)."""
import numpy as np

import bench
import oracle
from seed_hits_ungapped_gb300 import synth


def test_algorithmic_bytes_formula():
    # 16 B per seed, 13 B per anchor, both sequences once
    assert bench.algorithmic_bytes(10, 100, 1000, 50) == 16 * 10 + 13 * 100 + 1000 + 50
    assert bench.algorithmic_bytes(0, 0, 0, 0) == 0


def test_cpu_baseline_reports_rate_and_gate_pairs():
    w = synth.make("tiny", scale=0.2)
    cpu = bench.run_cpu_baseline(w, seconds=0.5)
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0
    ppa = cpu["gate_pairs_per_anchor"]
    # the sample's pairs per anchor equal the oracle's count over the same anchors
    idx, pos = oracle.build_index(w.ref)
    b = oracle.seed_buckets(w.query)
    P, total, rc = oracle.inclusive_prefix(oracle.count_hits(idx, b))
    T = oracle.keep_threshold(w.K)
    n_seeds = int(cpu["sample"].split("first ")[1].split(" seeds")[0])
    sub, s0 = [], 0
    while s0 < n_seeds:
        s1 = min(n_seeds, s0 + 200_000)
        hb = int(P[s0 - 1]) if s0 else 0
        a = oracle.expand(idx, pos, b, P, np.array([s0, s1, hb, P[s1 - 1]], np.uint32))
        sub.append(a[::16])
        s0 = s1
    sub = np.concatenate(sub)
    want = oracle.gate_pairs(w.ref, w.query, sub, w.matrix, w.xdrop, T) / len(sub)
    assert abs(ppa - want) < 1e-9
    # a seed anchor's decision scores at least its left walk through the seed
    assert ppa > 18


def test_kernel_hash_ignores_comments_only():
    src = 'int a = 1;  // walk\n/* step\n   block */\nconst char *s = "//x /*y*/";\nint b = a + 1;\n'
    assert bench.code_only(src) == 'int a = 1; const char *s = "//x /*y*/"; int b = a + 1;'
    assert bench.code_only(src.replace("// walk", "// other words")) == bench.code_only(src)
    assert bench.code_only(src.replace("a + 1", "a + 2")) != bench.code_only(src)


def test_clock_summary_keeps_samples_of_the_timed_region(tmp_path):
    """The clock record keeps the nvidia-smi samples whose timestamps fall in
    the timed region; a region shorter than the sampling interval takes the
    nearest sample."""
    import datetime
    path = tmp_path / "clocks.csv"
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5, 0)
    lines = []
    for i, (mhz, cap) in enumerate([(1400, "Active"), (2070, "Not Active"), (2070, "Not Active"),
                                    (1980, "Not Active"), (1200, "Active")]):
        ts = (t0 + datetime.timedelta(milliseconds=500 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        lines.append("%s, 0, %d, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, %s" % (ts, mhz, cap))
    path.write_text("\n".join(lines) + "\n")
    c = bench.ClockSampler(0, str(path))
    c.proc = object()  # as if nvidia-smi had run
    base = t0.timestamp()
    c.window = (base + 0.45, base + 1.55)  # samples 1, 2 and 3
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070 and s["reasons"] == [] and s["sampled"] == "timed region"
    c.window = (base + 2.2, base + 2.21)  # after the last sample (2.0 s): that one
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 1200 and s["reasons"] == ["sw_power_cap"]
    c.window = None
    s = c.summary()
    assert s["samples"] == 5 and s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070
