"""Host-side helpers of bench.py: the source digest that ties the DRAM-traffic
record to the kernels it was measured on, the clock-sample window, the bounded
oracle sample and the weak-scaling arithmetic.  No GPU."""
import json
import time

import pytest

import bench
import synthetic


def test_comment_stripping_keeps_code_and_literals():
    src = ('int a = 1; // note\n'
           '/* block\n comment */ const char* s = "a // b /* c */";\n'
           "char q = '\"'; char r = '/'; int b = 2 / 1; /* x */ int c;\n")
    got = bench.strip_c_comments(src)
    assert "note" not in got and "block" not in got and "x */" not in got
    assert '"a // b /* c */"' in got                 # comment markers inside a string stay
    assert "char q = '\"';" in got and "char r = '/';" in got
    assert "int b = 2 / 1;" in got and "int c;" in got
    assert bench.strip_c_comments("a/*unterminated") == "a"
    assert bench.strip_c_comments("int  a;\n\n  int b;  ") == "int a; int b;"


def test_digest_ignores_comments_but_not_code(tmp_path, monkeypatch):
    root = tmp_path
    (root / "moe_layer_serving_gb300" / "csrc").mkdir(parents=True)
    (root / "include").mkdir()
    kern = root / "moe_layer_serving_gb300" / "csrc" / "k.cu"
    hdr = root / "include" / "megamoe.h"
    kern.write_text("__global__ void k(int* p) { p[0] = 1; }  // stores one\n")
    hdr.write_text("/* C ABI */\nint f(void);\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    d0 = bench.sources_digest()
    kern.write_text("// the kernel\n__global__ void k(int* p) { p[0] = 1; }  // writes 1\n")
    hdr.write_text("/* the C ABI, reworded */\nint f(void);\n")
    assert bench.sources_digest() == d0
    kern.write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.sources_digest() != d0


def test_traffic_record_only_for_matching_sources(tmp_path, monkeypatch):
    root = tmp_path
    (root / "moe_layer_serving_gb300" / "csrc").mkdir(parents=True)
    (root / "include").mkdir()
    (root / "profiles").mkdir()
    (root / "moe_layer_serving_gb300" / "csrc" / "k.cu").write_text("int x;\n")
    (root / "include" / "megamoe.h").write_text("int f(void);\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    rec = {"small_kernel": {"w": {"bytes_per_launch": 123, "sources_sha256": bench.sources_digest()}}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.measured_traffic("small_kernel", "w") == 123
    assert bench.measured_traffic("small_kernel", "other") is None
    (root / "moe_layer_serving_gb300" / "csrc" / "k.cu").write_text("int y;\n")
    assert bench.measured_traffic("small_kernel", "w") is None


def test_clock_window_keeps_only_samples_inside_it():
    s = bench.ClockSampler(0)

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    class NoThread:
        def join(self, timeout=None):
            pass

    s.proc, s.thread = Done(), NoThread()
    idle = ["2070", "2070", "100", "Not Active", "Not Active", "Not Active", "Not Active"]
    busy = ["1700", "2070", "1390", "Not Active", "Not Active", "Not Active", "Active"]
    s.rows = [(1.0, idle), (2.0, busy), (3.0, busy), (4.0, idle)]
    sleep = time.sleep
    try:
        time.sleep = lambda _: None
        clk = s.stop(since=1.5, until=3.5)
    finally:
        time.sleep = sleep
    assert clk["samples"] == 2 and clk["sm_mhz"] == 1700.0 and clk["reasons"] == ["sw_power_cap"]


def test_bounded_oracle_sample_grows_then_repeats(monkeypatch):
    calls = []

    def fake(cfg, hidden, logits, bias, W, pmap, n, act="mxfp8", shared=0):
        n = min(n, cfg.T)
        calls.append(n)
        dt = 0.1 * n                    # 0.1 s per token
        return n / dt, dt, n

    monkeypatch.setattr(bench, "oracle_sample_rate", fake)
    cfg = synthetic.CONFIGS[1]          # T = 64
    rate, total, n, reps = bench.oracle_bounded_rate(cfg, None, None, None, None, None, 10.0)
    # 8 -> 0.8 s, 16 -> 1.6 s, 32 -> 3.2 s (>= 10 / 4): the sample stops growing at 32 tokens
    assert calls[:3] == [8, 16, 32] and n == 32
    assert total >= 10.0 and reps == 4 and rate == pytest.approx(10.0)
    calls.clear()
    cfg0 = synthetic.CONFIGS[0]         # T = 16: the whole batch, repeated at most 8 times
    _, total0, n0, reps0 = bench.oracle_bounded_rate(cfg0, None, None, None, None, None, 100.0)
    assert n0 == 16 and reps0 == 8 and total0 == pytest.approx(8 * 1.6)


def test_weak_scaling_value_counts_every_rank():
    assert bench.weak_scaling_value(64, 1, 0.5) == pytest.approx(128000.0)
    assert bench.weak_scaling_value(64, 4, 0.5) == pytest.approx(512000.0)


def test_scaled_down_workload_keeps_rows_per_expert_and_replica_share():
    full = synthetic.CONFIGS[4]
    small = bench.scaled_down(full, 8)
    assert (small.T, small.E, small.P) == (2048, 32, 40)
    assert small.T * small.k / small.E == full.T * full.k / full.E
    assert (small.P - small.E) / small.E == (full.P - full.E) / full.E
    assert (small.zipf_s, small.recording, small.H, small.I) == (full.zipf_s, full.recording, full.H, full.I)
    name = bench.workload_config(small)["workload"]
    assert name == "moe-layer-a8w4-T2048-E32-P40"
    assert bench.workload_config(full)["workload"] == "moe-layer-a8w4-T16384"
    with pytest.raises(SystemExit):
        bench.scaled_down(full, 3)


def test_routing_labels_name_the_recipe():
    assert bench.workload_config(synthetic.CONFIGS[1])["routing"] == "N(0,1) logits + N(0,0.1) selection bias"
    assert bench.workload_config(synthetic.CONFIGS[3])["routing"] == "N(0,1) logits"
    assert bench.workload_config(synthetic.CONFIGS[4])["routing"].startswith("zipf s=1.4")
