"""The benchmark's reference arm and its byte accounting, on the CPU: the JSON line carries
the contract's keys, and every workload's runner counts positive algorithmic bytes."""
import json
import os
import subprocess
import sys

import pytest

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", ["tiny_gqa_fp32"])
def test_reference_arm_json_line(name):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", name,
                        "--steps", "1", "--warmup", "1"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == name
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["unit"] == line["unit"]


def test_every_workload_has_a_runner_with_positive_bytes():
    sys.path.insert(0, ROOT)
    import bench
    for name, wl in W.WORKLOADS.items():
        assert wl.kind in bench.RUNNERS, name
    # describe() on small CPU inputs of each kind that has a cheap generator
    cfg, nbytes, flops = bench.GqaRunner.describe("tiny_gqa_fp32", W.build("tiny_gqa_fp32"))
    assert nbytes > 0 and flops > 0 and cfg["workload"] == "tiny_gqa_fp32"
    ring = W.make_ring(2, 8, 2, 64, [10, 5000], 256, n_sink=4, page_size=64, seed=2)
    cfg, nbytes, _ = bench.GqaRunner.describe("swa_ring_sink_tokens", ring)
    # a ring step reads the visible rows of both sequences plus the appended rows
    vis = 10 + (4 + 256)
    assert nbytes == vis * 2 * 64 * 2 * 2 + 2 * 2 * 2 * 2 * 64 * 2
    x = W.make_delta(4, 64, 32, seed=1)
    _, nbytes, _ = bench.DeltaRunner.describe("kda_decode", x)
    assert nbytes == 4 * (2 * 32 * 64 + 2 * 64 + 64 + 2 * 32 + 1) * 4
