"""The benchmark's reference arm on CPU: the oracle timed on the host cores
prints one JSON line with the fields the driver reads, and under a
multi-rank launch only rank 0 runs it (the other ranks exit 0 silently)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(env_extra: dict) -> subprocess.CompletedProcess:
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                           "--steps", "2", "--warmup", "3"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    res = run_reference({"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert res.returncode == 0, res.stderr
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_silently():
    res = run_reference({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""


def test_both_arms_share_one_config_block():
    """The driver compares the two arms' `config`: the encode arm's, for the
    default workload, must be exactly the reference arm's (timing details
    live under `timing`)."""
    import argparse

    sys.path.insert(0, ROOT)
    import bench
    import workloads

    for name in ("falcon_prefill", "tiny"):
        w = workloads.WORKLOADS[name]
        args = argparse.Namespace(partition=False, dtype="f16")
        ref = bench.config_block(w, args, 1)
        ours = dict(bench.config_block(w, args, 1), n_centroids=int(w.n_centroids),
                    input_dtype=args.dtype)
        assert ours == ref
        assert "l2" not in ref and "timed_region_s" not in ref
    res = run_reference({"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    d = json.loads(res.stdout.strip().splitlines()[-1])
    assert d["config"] == bench.config_block(workloads.WORKLOADS["tiny"],
                                             argparse.Namespace(partition=False), 1)
