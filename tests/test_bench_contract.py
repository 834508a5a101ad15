"""bench.py on the CPU: its command line, the reference arm's JSON line
(the reference arm times the oracle on the host), the profile keys and the
clock sampler's reading of nvidia-smi."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_defaults_are_one_gpu_and_minutes():
    sys.path.insert(0, ROOT)
    import bench

    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.variant == "sample"
    assert a.warmup >= 3 and a.steps >= 1


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key, kind in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                      ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                      ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[key], kind), key
    assert d["impl"] == "reference" and d["value"] > 0 and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_every_workload_is_a_bench_option_and_reference_arm_covers_it():
    """--workload takes each named workload; the reference arm's steps use
    that workload's rows (all of them when they fit the time budget)."""
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_verification_57_gb300 import workloads as W

    assert set(bench.WORKLOADS_DESC) == set(W.WORKLOADS)
    for name in W.WORKLOADS:
        assert bench.parse_args(["--workload", name]).workload == name
    assert bench.parse_args([]).workload == "benchmark"
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for name in ("toy", "zipf"):
        out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", name,
                              "--steps", "3", "--warmup", "1"], capture_output=True, text=True, cwd=ROOT, env=env,
                             timeout=600)
        assert out.returncode == 0, out.stderr[-2000:]
        d = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][0])
        w = W.make_workload(name)
        assert (d["config"]["B"], d["config"]["k"], d["config"]["V"]) == (w.B, w.k, w.V)
        assert d["config"]["rows_per_step"] == w.B


def test_profile_hash_ignores_comments():
    """A committed profile stays valid across comment edits, not code edits."""
    sys.path.insert(0, ROOT)
    import bench

    code = "int a = 1;  // note\n/* block\n comment */\nint b = 2;\n\n"
    assert bench._code_only(code) == "int a = 1;\nint b = 2;"
    assert bench._code_only(code.replace("note", "other note")) == bench._code_only(code)
    assert bench._code_only(code.replace("b = 2", "b = 3")) != bench._code_only(code)


def test_clock_sampler_keeps_the_timed_window_and_reasons(monkeypatch):
    """nvidia-smi rows outside the timed window are left out, the median SM
    clock and the active throttle reasons come from the rows inside it."""
    import time

    sys.path.insert(0, ROOT)
    import bench

    rows = [
        "2026/12/02 15:00:00.000, 0, 1500, 2070, 500.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 15:00:01.000, 0, 2070, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 15:00:01.100, 0, 2055, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 15:00:01.200, 0, 2070, 2070, 960.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 15:00:03.000, 0, 1000, 2070, 300.0, 0x8, Active, Not Active, Not Active, Not Active",
        "not a sample",
    ]

    class FakeSmi:
        def terminate(self):
            pass

        def kill(self):
            pass

        def communicate(self, timeout=None):
            return "\n".join(rows), ""

    monkeypatch.setattr(bench.subprocess, "Popen", lambda *a, **k: FakeSmi())
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    cs = bench.ClockSampler(0)
    cs.start()
    cs.t0 = time.mktime(time.strptime("2026/12/02 15:00:01", "%Y/%m/%d %H:%M:%S"))
    cs.t1 = cs.t0 + 0.2
    d = cs.stop()
    assert d["in_window"] and d["samples"] == 3
    assert d["sm_mhz"] == 2070.0 and d["sm_max_mhz"] == 2070.0
    assert d["reasons"] == ["sw_power_cap"]  # the hw_slowdown row lies outside the window


def test_filter_flags_and_profile_keys(monkeypatch):
    """--top-k / --top-p reach the filtered variant (defaults 40 / 0.95);
    the small-vocabulary kernel named in a profile key is the one the
    library picks for the batch (one CTA per row up to twice the SM count,
    SPECV_SMALLV forcing either), and every profile key has its sources."""
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_verification_57_gb300 import workloads as W

    a = bench.parse_args(["--variant", "filtered", "--top-k", "4096", "--top-p", "0.9"])
    assert (a.variant, a.top_k, a.top_p) == ("filtered", 4096, 0.9)
    b = bench.parse_args(["--variant", "filtered"])
    assert b.top_k is None and b.top_p is None and (bench.FILTER_TOP_K, bench.FILTER_TOP_P) == (40, 0.95)
    monkeypatch.delenv("SPECV_SMALLV", raising=False)
    assert bench.small_v_kernel(1, 152) == "verify_row_kernel"
    assert bench.small_v_kernel(304, 152) == "verify_row_kernel"
    assert bench.small_v_kernel(305, 152) == "verify_warp_kernel"
    monkeypatch.setenv("SPECV_SMALLV", "warp")
    assert bench.small_v_kernel(1, 152) == "verify_warp_kernel"
    monkeypatch.delenv("SPECV_SMALLV")
    toy = W.make_workload("toy")
    assert bench.profile_name("toy", toy) in bench.KERNEL_SOURCES
    assert bench.measured_traffic("no_such_profile") is None
    for name, files in bench.KERNEL_SOURCES.items():
        assert os.path.exists(os.path.join(ROOT, "profiles", name + ".md")), name
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "speculative_decoding_verification_57_gb300", "csrc", f)), f
