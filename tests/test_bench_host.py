"""Host-side logic of bench.py (no GPU): the nvidia-smi clock summary that
the line's `clocks` key comes from, and the reference arm's JSON line."""
import datetime
import importlib.util
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _line(t, sm, smax, hw="Not Active", hwt="Not Active", swt="Not Active", pc="Not Active"):
    return (f"{t.strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, 0, {sm}, {smax}, 900.00, 0x0, "
            f"{hw}, {hwt}, {swt}, {pc}\n")


def test_clock_summary_takes_the_timed_window():
    b = _bench()
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    lines = [_line(t0 - 500 * ms, 1200, 2070, hw="Active"),            # before the region
             _line(t0 + 10 * ms, 2070, 2070),
             _line(t0 + 60 * ms, 2055, 2070, pc="Active"),
             _line(t0 + 110 * ms, 2070, 2070),
             "garbage line\n",
             _line(t0 + 900 * ms, 600, 2070, swt="Active")]            # after the region
    s = b.clock_summary(lines, (t0, t0 + 120 * ms))
    assert s["samples"] == 3 and s["in_timed_region"] is True
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]       # the slowdowns outside the window are not counted


def test_clock_summary_falls_back_to_all_samples():
    b = _bench()
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = datetime.timedelta(milliseconds=1)
    lines = [_line(t0, 1500, 2070, hwt="Active"), _line(t0 + 50 * ms, 1700, 2070)]
    far = (t0 + 5000 * ms, t0 + 6000 * ms)
    s = b.clock_summary(lines, far)
    assert s["in_timed_region"] is False and s["samples"] == 2
    assert s["sm_mhz"] == 1600.0 and s["reasons"] == ["hw_thermal_slowdown"]
    assert b.clock_summary(["nonsense\n"], far) is None
    assert b.clock_summary([], None) is None


def test_reference_arm_line_keeps_the_contract():
    import oracle
    oracle.build()
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--workload", "bert_large_ffn_up_m256",
                        "--reference-step-seconds", "0.05"], cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["unit"] == "TOPS" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "bert_large_ffn_up_m256"
    assert set(d["cpu_baseline"]) >= {"value", "unit", "cores", "kind", "sample"}
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TOPS", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_refused():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--warmup", "2"], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert p.returncode != 0 and "warmup" in p.stderr
