"""The reference arm of the benchmark (`bench.py --impl reference`), run as the driver runs
it: the fp64 oracle timed on the host cores, one JSON line with the same metric, unit and
direction as the GPU arm.  It needs no GPU, so it is checked here end to end with a short
per-step budget."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(workload):
    env = dict(os.environ, GQA_REF_STEP_SECONDS="0.2")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          workload, "--steps", "2", "--warmup", "3"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,unit", [("plamo3_local_prefill", "TFLOP/s"),
                                           ("plamo3_decode_batch32", "GB/s")])
def test_reference_arm_line(workload, unit):
    d = _run(workload)
    assert d["impl"] == "reference"
    assert d["unit"] == unit and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == workload
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == unit
    assert cb["cores"] == os.cpu_count() and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == unit
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert d["ms_per_step"] > 0
