"""The benchmark's host logic on CPU.

The clock record decides whether a bench run is accepted (the median SM
clock under load and every throttle reason seen in the timed region), so its
parsing and the sampler's start-up are checked here against stand-in
nvidia-smi output.  The reference arm (the oracle timed on the host cores)
runs end to end and must print the bench's JSON line.
"""
import json
import os
import subprocess
import sys
import tempfile

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NA = "Not Active"


class _Proc:
    """Stands in for the nvidia-smi process."""

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _line(sm, smax=2070, reasons=(NA, NA, NA, NA)):
    # index, clocks.sm, clocks.max.sm, power.draw, clocks_event_reasons.active,
    # then hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return ", ".join(["0", str(sm), str(smax), "950.00", "0x0000000000000000", *reasons])


def _sampler_with(lines):
    s = bench.ClockSampler(0)
    fd, s.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("".join(x + "\n" for x in lines))
    s.fh = open(os.devnull, "w")
    s.proc = _Proc()
    return s


def test_clock_record_median_and_no_reason():
    rec = _sampler_with([_line(2070), _line(2070), _line(1980)]).stop()
    assert rec == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": []}


def test_clock_record_names_every_active_reason():
    rec = _sampler_with([
        _line(2070),
        _line(1500, reasons=("Active", NA, NA, NA)),
        _line(1400, reasons=(NA, "Active", "Active", "Active")),
    ]).stop()
    assert rec["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap",
                              "sw_thermal_slowdown"]
    assert rec["sm_mhz"] == 1500.0 and rec["samples"] == 3


def test_clock_record_skips_unreadable_lines():
    rec = _sampler_with([_line("[N/A]"), "garbage", _line(2055, smax=2070)]).stop()
    assert rec["samples"] == 1 and rec["sm_mhz"] == 2055.0


def test_clock_record_without_samples():
    rec = _sampler_with([]).stop()
    assert rec["sm_mhz"] is None and rec["reasons"] == ["no samples"]


def test_sampler_falls_back_to_50_ms(monkeypatch):
    """An nvidia-smi that writes nothing at a 10 ms interval: the sampler
    starts again at 50 ms and waits until that one produces a sample."""
    tried = []

    class FakePopen(_Proc):
        def __init__(self, args, stdout=None, stderr=None):
            interval = args[args.index("-lms") + 1]
            tried.append(interval)
            if interval == "50":
                stdout.write(_line(2070) + "\n")
                stdout.flush()

    monkeypatch.setattr(bench.subprocess, "Popen", FakePopen)
    s = bench.ClockSampler(0)
    s.start()
    assert tried == ["10", "50"]
    rec = s.stop()
    assert rec["samples"] == 1 and rec["reasons"] == []


def test_reference_arm_prints_the_bench_line():
    """`bench.py --impl reference` with a short per-step budget: one JSON line
    with the bench's keys, the oracle's rate as value, cpu_baseline and e2e."""
    r = subprocess.run(
        [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
         "--ref-step-seconds", "0.5"],
        cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["metric"] == "sparse-MLA fwd+bwd TFLOPS" and d["unit"] == "TFLOP/s"
    assert "flash_t8k" in d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
