"""`bench.py --impl reference` (the oracle arm, host cores only, no GPU): one
JSON line with the driver's keys, the same metric, unit and `config` record
as the GPU arm prints for the workload, and a bounded sample."""
import json
import os
import subprocess
import sys
import types

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "1"], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tok/s"
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 1
    assert d["value"] > 0
    # the config the GPU arm prints for the default workload and these flags
    args = types.SimpleNamespace(workload="smollm2-135m-bf16", layers=0, warmup=1, steps=1)
    assert d["config"] == bench.workload_config(args, bench.WORKLOADS[args.workload], 256, 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "32 of 256 lanes" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tok/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
