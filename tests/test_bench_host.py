"""Host side of bench.py on CPU: the reference arm's JSON line (the oracle timed
on host cores, with the keys the line must carry) and the refusal of options
that do not apply (a near window outside 32..64, or above 32 on a level-1
workload or in split mode)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT)


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["warmup"] >= 3
    assert line["config"]["workload"] == "tiny_256x256_u32"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_window_line():
    r = _bench("--impl", "reference", "--config", "1", "--window", "64", "--steps", "1",
               "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["config"]["near_window"] == 64


def test_window_options_refused():
    for args in (("--window", "31"), ("--window", "65"), ("--window", "48", "--config", "3"),
                 ("--window", "48", "--split")):
        r = _bench("--impl", "reference", *args, timeout=120)
        assert r.returncode != 0, args
        assert "--window" in (r.stderr + r.stdout), args
