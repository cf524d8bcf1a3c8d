"""The benchmark's reference arm (the fp64 oracle on the host cores) prints
one JSON line with the contract's keys; it needs no GPU, so it runs here."""
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
