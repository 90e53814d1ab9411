"""bench.py --impl reference on the CPU: the oracle timed on the host cores,
one JSON line with the contract's keys, and a run time bounded by
--ref-seconds whatever --steps is (on the one-head workload C2, so that
the inputs are quick to make)."""
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*extra):
    t0 = time.perf_counter()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "C2", *extra], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0]), time.perf_counter() - t0


def test_reference_line_keys():
    line, _ = _run("--steps", "3", "--warmup", "3", "--ref-rows", "64")
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3
    assert line["unit"] == "TFLOPS" and line["higher_is_better"] is True and line["value"] > 0
    assert line["config"]["workload"] == "C2_b1h1n4096d64_fp16"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert cb["sample"].startswith("64 seeded query rows")
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_many_steps_stay_within_the_time_bound():
    """1000 steps with a 2-second bound: each step shrinks to a row or a few,
    on the threads such a sample keeps busy, instead of the run growing with
    the step count."""
    line, wall = _run("--steps", "1000", "--warmup", "3", "--ref-seconds", "2")
    assert line["steps"] == 1000 and line["value"] > 0
    rows = int(line["cpu_baseline"]["sample"].split()[0])
    assert rows < 256 and line["cpu_baseline"]["cores"] == max(
        1, min(len(os.sched_getaffinity(0)), -(-rows // 16)))
    assert wall < 90, wall
