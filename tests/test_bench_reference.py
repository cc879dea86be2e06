"""bench.py's reference arm (the oracle timed on the host cores) prints the contract's
JSON line; it needs no GPU, so it runs here on small samples of two workloads."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


@pytest.mark.parametrize("extra,unit", [(["--workload", "single_stream", "--rounds", "2"], "verify rows/s"),
                                        (["--workload", "tree_mask", "--batch", "8", "--nodes", "60"], "trees/s")])
def test_reference_arm_prints_the_contract_line(extra, unit):
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3", *extra],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert REQUIRED <= set(line)
    assert line["impl"] == "reference" and line["unit"] == unit and line["value"] > 0
    assert line["higher_is_better"] is True and line["data"] == "synthetic"
    assert line["steps"] == 2 and line["warmup"] >= 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == unit
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"]


def test_both_arms_print_the_same_config():
    """The reference arm's `config` is the one the GPU arm prints for the same workload
    (both come from one function of the workload), so the two lines compare like for like."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                          "--workload", "single_stream", "--rounds", "2"], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["config"] == bench.workload_config(bench.make_workload("single_stream", 0, 2), 1)
    args = argparse.Namespace(workload="tree_mask", batch=8, nodes=60, steps=1)
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                          "--workload", "tree_mask", "--batch", "8", "--nodes", "60"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["config"] == bench.aux_config(bench.make_aux(args, 0), 1)


def test_large_batch_at_another_temperature_is_one_workload():
    """The large batch at T != 0.7 is the T = 0.7 logits with the drafts redrawn at T,
    whether it is the run's workload or a side line, so one ncu summary per temperature
    describes both; each such summary names its own temperature."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    base = bench.make_workload("large_batch", 0, 64, batch=2, temperature=0.7)
    for T in (0.0, 1.5):
        run = bench.make_workload("large_batch", 0, 64, batch=2, temperature=T)
        side = bench.large_batch_at(base, T)
        for k in ("target", "draft", "tokens", "temperature"):
            assert np.array_equal(run[k], side[k]), (T, k)
        assert (run["temperature"] == np.float32(T)).all()
        traffic, path, kernel = bench.profile_traffic(f"large_batch_T{T:g}")
        assert path is not None and path.endswith(f"_large_batch_T{T:g}.md") and kernel == "chain_staged_kernel"
    assert bench.large_batch_at(base, 0.7) is base
