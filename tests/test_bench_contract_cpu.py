"""Host-side pieces of bench.py's JSON contract, on CPU: the reference arm's line
(the oracle timed on the host cores, with its cpu_baseline and a zero-copy e2e)
and the clock summary of the timed region (median SM clock, throttle reasons,
samples outside the window dropped)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_the_contract_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("block3b")


def test_clock_summary_uses_the_timed_window_and_reports_reasons():
    import bench
    c = bench.ClockSampler(0)
    c.lines = [(0.0, "900, 2070, 300, Not Active, Not Active, Not Active, Not Active"),    # before the window
               (1.0, "2070, 2070, 1200, Not Active, Not Active, Not Active, Active"),
               (1.1, "2040, 2070, 1300, Not Active, Not Active, Not Active, Active"),
               (1.2, "2070, 2070, 1250, Not Active, Not Active, Not Active, Not Active"),
               (5.0, "1000, 2070, 1250, Active, Not Active, Not Active, Not Active")]          # after it
    c.window = (0.95, 1.25)
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c.window = (4.9, 5.1)
    assert c.summary()["reasons"] == ["hw_slowdown"]
    c.lines = []
    assert c.summary()["reasons"] == ["unsampled"]
