"""CPU checks of bench.py: the JSON line of the reference arm (the CPU oracle
timed on the host on a bounded sample of the benchmark step) and the hash
that ties the committed DRAM-traffic capture to the kernel code."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["unit"] == "TOPS" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "prefill_27b_w8a8"
    assert d["config"]["shapes"] == [[8192, 5120, 17408], [8192, 17408, 5120]]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] and cb["unit"] == d["unit"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_capture_hash_follows_code_not_comments(tmp_path):
    import bench
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) { return x + 1; }  // one more\n/* a block\n comment */\n")
    b = tmp_path / "b.cu"
    b.write_text("// header comment\nint f(int x) {\n  return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.source_sha(str(a)) == bench.source_sha(str(b))
    assert bench.source_sha(str(a)) != bench.source_sha(str(c))
    assert bench.sources_sha([str(a), str(c)]) != bench.sources_sha([str(c), str(a)])


def test_clock_summary_keeps_the_timed_window():
    """The clock record keeps the samples inside the timed region when there
    are enough of them, reports throttle reasons seen there, and falls back
    to all samples (warm-up included) otherwise."""
    import bench
    import datetime
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5).timestamp()

    def line(dt, mhz, power_cap):
        stamp = datetime.datetime.fromtimestamp(t0 + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        cap = "Active" if power_cap else "Not Active"
        return "%s, 0, %d, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, %s" % (stamp, mhz, cap)

    c = bench.ClockSampler(0)
    c.lines = [line(0.00, 1500, True), line(0.10, 2000, False), line(0.15, 2010, False),
               line(0.20, 2020, False), line(0.50, 1400, True)]
    s = c.summary((t0 + 0.05, t0 + 0.3))
    assert s["samples"] == 3 and s["sm_mhz"] == 2010 and s["reasons"] == []
    assert s["window"] == "timed region"
    s = c.summary((t0 + 0.05, t0 + 0.12))          # one sample inside: all samples
    assert s["samples"] == 5 and "sw_power_cap" in s["reasons"]
