"""bench.py on the CPU: every workload name builds, and the reference arm
(the oracle on host cores) prints one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_every_workload_name_builds(name):
    wl, layout, shared = bench.make_workload(*bench.WORKLOADS[name])
    assert wl.num_seqs > 0 and layout in ("row", "split") and shared in (True, False)


def test_reference_arm_prints_one_contract_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "cfg0",
           "--steps", "3", "--warmup", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"]
    assert d["steps"] == 3 and d["warmup"] == 1 and d["n_gpus"] == 1 and d["gpu_launches"] == 0
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["cores"] >= 1 and cpu["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "cfg0",
           "--steps", "3", "--warmup", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""


def test_reference_arm_config_is_the_gpu_arms_config():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "cfg0",
           "--steps", "2", "--warmup", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    d = json.loads(res.stdout.strip().splitlines()[-1])
    wl, _, _ = bench.make_workload(*bench.WORKLOADS["cfg0"])  # rank 0 of the GPU arm: no seed offset
    assert d["config"] == json.loads(json.dumps(bench.bench_config(wl, "none", 1)))


def test_clock_sampler_says_why_it_has_no_samples():
    """Without a GPU (here) the sampler neither raises nor invents a clock:
    its record has no samples and a reason."""
    s = bench.ClockSampler(0)
    s.start()
    rec = s.stop()
    if rec["samples"] == 0:
        assert rec["sm_mhz"] is None and rec["why_none"]
    else:  # a machine with a readable GPU
        assert rec["sm_mhz"] > 0 and rec["source"]
