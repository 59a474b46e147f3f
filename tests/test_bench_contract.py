"""bench.py's command line and JSON line, checked on the CPU through its reference arm.

The reference arm times the float64 oracle on a token sample on the host cores, so it runs
without a GPU; these tests run it on the tiny workload and check the line's keys and values,
that non-zero ranks stay silent, and that fewer than three warm-up steps are refused.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BENCH = os.path.join(ROOT, "bench.py")


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, BENCH] + args, cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
              "--oracle-tokens", "16"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # tokens per second over the timed steps: 16 tokens per step
    assert abs(d["value"] - 16 * 1e3 / d["ms_per_step"]) <= 1e-6 * d["value"]
    assert d["config"]["workload"] == "tiny"
    assert d["config"]["tokens"] == 128 and d["config"]["vocab"] == 2048
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "16 tokens" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_is_silent_on_other_ranks():
    r = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"],
             {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_fewer_than_three_warmup_steps_are_refused():
    r = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "2"])
    assert r.returncode == 2
    assert "--warmup must be >= 3" in r.stderr


def test_cpu_baseline_times_at_least_the_bounded_duration():
    """The CPU baseline repeats token samples of the workload until its minimum duration has
    passed and reports tokens per second over all of them."""
    sys.path.insert(0, ROOT)
    import bench
    from lm_head_linear_02_gb300.inputs import make_inputs

    inp = make_inputs("tiny")
    cb = bench.cpu_baseline(inp, 48, min_seconds=0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["cores"] >= 1
    done = int(cb["sample"].split()[0])
    secs = float(cb["sample"].rsplit(",", 1)[1].split()[0])
    assert done >= 48 and done % 48 == 0 and "samples of 48" in cb["sample"]
    elapsed = done / cb["value"]
    assert elapsed >= 0.3
    assert abs(elapsed - secs) <= 0.051  # the sample text prints the seconds to 0.1


def test_tuning_arguments_parse_and_refuse_unknown_names():
    import bench

    assert bench.parse_tuning(["raster_vocab=4096", "chunk_bytes=0x40000000"]) == {
        "raster_vocab": 4096, "chunk_bytes": 1 << 30}
    for bad in (["raster_vocab"], ["nonsense=1"], ["raster_vocab=abc"]):
        with pytest.raises(ValueError):
            bench.parse_tuning(bad)


def test_clock_sampler_keeps_the_timed_window_and_reports_power():
    """The nvidia-smi sampler keeps the rows stamped inside the timed window: median SM clock,
    maximum clock, the throttle reasons seen active, and the median board power (rows whose
    power reads "[N/A]" are left out of that median)."""
    import datetime

    sys.path.insert(0, ROOT)
    import bench

    def stamp(sec):
        return datetime.datetime.fromtimestamp(sec).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]

    t0 = 1_800_000_000.0
    rows = [
        (t0 - 1.0, 2070, 400.0, "Not Active"),  # before the window
        (t0 + 0.1, 1600, 1390.0, "Active"),
        (t0 + 0.2, 1620, 1380.0, "Active"),
        (t0 + 0.3, 1640, None, "Active"),
        (t0 + 5.0, 2070, 300.0, "Not Active"),  # after the window
    ]
    text = "\n".join(
        f"{stamp(ts)}, {sm}, 2070, {'[N/A]' if pw is None else pw}, 0x4, Not Active, Not Active, "
        f"Not Active, {cap}" for ts, sm, pw, cap in rows)

    class FakeProc:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            return text, ""

    s = bench.ClockSampler(0)
    s.proc = FakeProc()
    s.t0, s.t1 = t0, t0 + 1.0
    out = s.stop()
    assert out["in_timed_window"] and out["samples"] == 3
    assert out["sm_mhz"] == 1620 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w"] == pytest.approx(1385.0)
