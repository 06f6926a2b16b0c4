"""Host-side pieces of bench.py: the code identity used for the DRAM-traffic
lookup."""
import bench


def test_code_tokens_ignore_comments_and_layout_only():
    a = 'int f(int x) {\n  // a comment\n  return x + 1; /* block\n comment */\n}\n'
    b = 'int f(int x){return x+1;}'
    assert bench.code_tokens(a) == bench.code_tokens(b)
    assert bench.code_tokens('return x + 2;') != bench.code_tokens('return x + 1;')
    # "//" inside a string literal is code, not a comment
    assert bench.code_tokens('const char* s = "a//b";') == 'constchar*s="a//b";'
    assert bench.code_tokens('x = "a\\"//";') == 'x="a\\"//";'


def test_every_kernel_has_a_code_hash():
    for k in bench.KERNEL_SOURCES:
        assert len(bench.source_hash(k)) == 16


def test_traffic_entries_are_reported_only_for_the_code_they_were_taken_on():
    import json
    import os
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for kernel, workloads in t.items():
        if kernel.startswith("_"):
            continue
        assert kernel in bench.KERNEL_SOURCES, kernel
        for workload, e in workloads.items():
            assert e["bytes_per_launch"] == e["read"] + e["write"], (kernel, workload)
            assert len(e["source_hash"]) == 16
            current = e["source_hash"] == bench.source_hash(kernel)
            got = bench.dram_traffic(kernel, workload)
            assert got == (e["bytes_per_launch"] if current else None), (kernel, workload)
    assert bench.dram_traffic("prefill_kernel", "no such workload") is None


def test_cpu_baseline_extras_report_the_documented_fields():
    extras = bench.cpu_baseline_extras(0.05)
    assert [e["workload"] for e in extras] == ["prefill_b4_s1024_h16_kv8",
                                              "decode_n256_len128to2048_h16_kv8"]
    assert extras[0]["cores"] == 1 and extras[0]["unit"] == "TFLOP/s"
    assert extras[1]["unit"] == "GB/s" and extras[1]["cores"] >= 1
    assert all(e["value"] > 0 and e["sample"] for e in extras)


def test_reference_arm_prints_one_contract_line():
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--cpu-seconds", "0.5"], cwd=bench.ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_clock_summary_keeps_only_samples_inside_the_timed_region(tmp_path):
    """The clocks line reports samples stamped inside the timed window, with their
    throttle reasons; a window that no sample falls in falls back to the whole run."""
    import datetime
    import time as _time

    class _Done:
        def terminate(self):
            pass

        def wait(self):
            pass

    def sampler(rows):
        c = bench.ClockSampler.__new__(bench.ClockSampler)
        path = tmp_path / f"clk{len(rows)}_{_time.monotonic_ns()}.csv"
        path.write_text("".join(rows))
        c.f = open(path, "r+")
        c.p = _Done()
        return c

    now = _time.time()
    rows = []
    for k, (mhz, cap) in enumerate([(1500, "Not Active"), (2070, "Not Active"),
                                    (2040, "Not Active"), (1900, "Active")]):
        stamp = datetime.datetime.fromtimestamp(now + 0.02 * k).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        rows.append(f"{stamp}, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}\n")
    inside = sampler(rows).stop((now + 0.01, now + 0.05))
    assert inside["samples"] == 2 and inside["samples_run"] == 4
    assert inside["window"] == "timed region"
    assert inside["sm_mhz"] == 2055.0 and inside["reasons"] == []
    outside = sampler(rows).stop((now + 10.0, now + 11.0))
    assert outside["window"] == "whole run" and outside["samples"] == 4
    assert outside["reasons"] == ["sw_power_cap"]
