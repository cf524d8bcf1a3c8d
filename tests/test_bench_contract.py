"""The benchmark's host-side parts: the reference arm (the fp64 oracle on
the host cores) prints one JSON line with the contract's keys, and the clock
sampler turns nvidia-smi rows into the median SM clock and the throttle
reasons a run is judged by.  Neither needs a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_line(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny", "--steps", "2",
           "--warmup", "3", "--reference-seconds", "1", *extra]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("extra", [(), ("--backward",)])
def test_reference_arm_prints_the_contract_line(extra):
    j = _reference_line(*extra)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference"
    assert j["steps"] == 2 and j["warmup"] == 3 and j["higher_is_better"] is True
    assert j["value"] > 0 and j["unit"] == "TFLOP/s" and j["dtype"] == "f64"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["d2h_bytes_per_step"] == 0
    assert ("bwd" in j["metric"]) == bool(extra)


class _DoneProc:
    """A finished nvidia-smi process: its lines are already read."""

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_samples_parse_to_median_and_reasons():
    # rows as nvidia-smi --format=csv,noheader,nounits prints the sampler's
    # fields: index, SM clock, max SM clock, power, active mask, then the four
    # throttle reasons the rejection rule names
    import bench
    cs = bench.ClockSampler(0)
    cs.proc = _DoneProc()
    cs.lines = ["0, 1845, 2032, 1050.2, 0x4, Not Active, Not Active, Not Active, Active",
                "0, 2017, 2032, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active",
                "0, 1530, 2032, 1099.9, 0x4, Not Active, Not Active, Not Active, Active",
                "[N/A], [N/A]",                                   # a malformed row is skipped
                "0, [N/A], 2032, 0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    got = cs.stop()
    assert got == {"sm_mhz": 1845.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"], "samples": 3}
    cs.lines = ["0, 900, 2032, 700.0, 0x48, Active, Not Active, Active, Not Active"]
    assert cs.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_sampler_without_nvidia_smi():
    import bench
    got = bench.ClockSampler(0).stop()     # never started: no process
    assert got["sm_mhz"] is None and got["reasons"] == ["nvidia-smi unavailable"]
