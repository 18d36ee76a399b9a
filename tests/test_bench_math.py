"""The bench's measurement arithmetic, on the host: the host-link busy time
(union of the gather launches' intervals), algorithmic GB/s and the fraction
of each kind's peak, and the lookup of recorded DRAM traffic, which must go
null once the kernel's source changes."""
import random

import bench


def _cells(intervals):
    # brute force on integer endpoints: unit cells covered by any interval
    return sum(1 for c in range(0, 200) if any(a <= c < b for a, b in intervals))


def test_link_busy_is_the_union_of_gather_intervals():
    assert bench.link_busy_ms([]) == 0.0
    assert bench.link_busy_ms([("ffn", 0.0, 5.0)]) == 0.0
    g = lambda *iv: [("gather", a, b) for a, b in iv]  # noqa: E731
    assert bench.link_busy_ms(g((0, 2), (1, 3))) == 3        # overlap
    assert bench.link_busy_ms(g((0, 1), (2, 4))) == 3        # disjoint
    assert bench.link_busy_ms(g((0, 5), (1, 2))) == 5        # nested
    assert bench.link_busy_ms(g((0, 1), (1, 2))) == 2        # touching
    assert bench.link_busy_ms(g((2, 4), (0, 1)) + [("set", 0, 9)]) == 3  # order, other kinds
    rng = random.Random(7)
    for _ in range(200):
        iv = []
        for _ in range(rng.randint(1, 12)):
            a = rng.randint(0, 150)
            iv.append((a, a + rng.randint(0, 40)))
        assert bench.link_busy_ms(g(*iv)) == _cells(iv)


def test_kernel_table_rates_and_fractions():
    prof = {"ffn": {"launches": 4, "ms": 0.1, "bytes": 4 * 50_000_000},
            "gather": {"launches": 2, "ms": 1.0, "bytes": 200_000_000},
            "set": {"launches": 0, "ms": 0.0, "bytes": 0},
            "finish": {"launches": 3, "ms": 0.015, "bytes": 0}}
    t = bench.kernel_table(prof, {"hbm_gbs": 6800.0}, 200.0)
    assert "set" not in t
    ffn = t["ffn"]
    assert ffn["bound"] == "hbm" and ffn["gbs"] == 2000.0 and ffn["us_per_launch"] == 25.0
    assert ffn["bytes_per_launch"] == 50_000_000 and abs(ffn["frac"] - 2000.0 / 6800.0) < 1e-4
    ga = t["gather"]
    assert ga["bound"] == "host_link" and ga["gbs"] == 200.0 and ga["frac"] == 1.0
    assert t["finish"]["gbs"] is None and t["finish"]["frac"] is None


def test_recorded_traffic_needs_the_captured_source(monkeypatch):
    cur = bench.file_hash(bench.os.path.join(bench.SRC_DIR, "np_ffn.cu"))
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {
        ("ffn", "w"): {"src": "np_ffn.cu", "src_hash": cur, "bytes_per_launch": 123},
        ("dense", "w"): {"src": "np_ffn.cu", "src_hash": "0" * 16, "bytes_per_launch": 456}})
    assert bench.traffic_for("ffn", "w") == 123
    assert bench.traffic_for("dense", "w") is None      # kernel changed since the capture
    assert bench.traffic_for("ffn", "other") is None    # never captured


def test_recorded_traffic_entries_name_existing_sources():
    for (kind, workload), ent in bench.NCU_TRAFFIC.items():
        assert bench.os.path.exists(bench.os.path.join(bench.SRC_DIR, ent["src"])), (kind, workload)
        assert len(ent["src_hash"]) == 16 and ent["bytes_per_launch"] > 0


def test_clock_summary_parses_nvidia_smi_lines():
    cs = bench.ClockSampler(0)
    cs.lines = ["2070, 2070, 812.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
                "1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
                "garbage line",
                "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
                "2040, 2070, 1100.1, 0x0000000000000008, Active, Not Active, Not Active, Not Active"]
    s = cs.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2040.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(0).summary()
    assert empty == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_link_overlap_against_brute_force():
    # exposed link time = link busy with no compute kernel running; idle =
    # compute with the link idle; checked on a fine time grid
    import random
    import bench
    rnd = random.Random(7)
    for _ in range(20):
        tl = []
        for _ in range(rnd.randint(1, 12)):
            k = rnd.choice(["gather", "gather", "ffn", "dense", "predictor", "set", "finish", "scatter"])
            a = rnd.randint(0, 200) / 10
            tl.append((k, a, a + rnd.randint(1, 60) / 10))
        ov = bench.link_overlap(tl)
        step = 0.01
        grid = [i * step + step / 2 for i in range(int(30 / step))]
        on = lambda kinds, t: any(a <= t < b for k, a, b in tl if k in kinds)
        link = sum(step for t in grid if on(("gather",), t))
        comp = sum(step for t in grid if on(bench.COMPUTE_KINDS, t))
        both = sum(step for t in grid if on(("gather",), t) and on(bench.COMPUTE_KINDS, t))
        assert abs(ov["busy"] - link) < 0.05
        assert abs(ov["exposed"] - (link - both)) < 0.05
        assert abs(ov["idle_while_compute"] - (comp - both)) < 0.05
