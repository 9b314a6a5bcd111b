"""The JSON line of bench.py's reference arm (the float64 oracle on the host
cores), checked on the CPU: one line, the same metric, unit, direction and
workload description as the GPU arm, the oracle named as its kind, and an
end-to-end figure with no host-device copies."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ref_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_line_keys(ref_line):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in ref_line, key
    assert ref_line["impl"] == "reference"
    assert ref_line["value"] > 0 and ref_line["ms_per_step"] > 0
    assert ref_line["steps"] == 1 and ref_line["warmup"] == 3 and ref_line["n_gpus"] == 1
    assert ref_line["data"] == "synthetic" and ref_line["dtype"] == "f64"
    cb = ref_line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == ref_line["value"] and cb["cores"] >= 1
    assert cb["unit"] == ref_line["unit"] and cb["sample"]
    e2e = ref_line["e2e"]
    assert e2e == {"value": ref_line["value"], "unit": ref_line["unit"], "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}


def test_reference_line_matches_the_gpu_arm(ref_line):
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    wl = workloads.named(bench.DECODE)
    assert ref_line["metric"] == bench.HEADLINE_METRIC
    assert ref_line["unit"] == "GB/s" and ref_line["higher_is_better"] is True
    assert ref_line["scaling"] == "weak" and ref_line["vs_baseline"] is None
    assert ref_line["config"] == bench.headline_config(workloads, wl, 1)


@pytest.mark.parametrize("index,launches", [(1, 2), (2, 2), (3, 2), (4, 2), (5, 3)])
def test_launch_count_claim_follows_the_launch_rules(index, launches):
    # the line's gpu_launches claim: the plan, then the decode kernel only when
    # some unit may hold <= 16 packed rows (not when every sequence must hold
    # more than 16 / G queries: the tiny decode's 8-query sequences at G 6, the
    # prefill batches), and the prefill kernel only when some unit may hold more
    # (not the decode batch's 1-query sequences at G 4)
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    assert bench.launches_per_step(workloads.named(index, scale_down=1 if index < 3 else 16)) == launches
