"""The benchmark's reference arm (the fp64 oracle on host cores) needs no GPU:
its one JSON line carries the contract's keys, only rank 0 prints under a
multi-rank launch, and too few warm-up steps are rejected."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=300)


def test_reference_line_has_the_contract_keys():
    import bench

    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3", "--workload",
              "b1h1n256d64"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference"
    assert out["metric"] == bench.METRIC and out["unit"] == bench.UNIT
    assert out["value"] > 0 and out["ms_per_step"] > 0
    assert (out["n_gpus"], out["steps"], out["warmup"]) == (1, 3, 3)
    assert out["higher_is_better"] is True and out["scaling"] == "weak"
    assert out["vs_baseline"] is None and out["dtype"] == "f64" and out["data"] == "synthetic"
    assert out["config"]["workload"] == "b1h1n256d64"
    cpu = out["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == out["value"]
    assert cpu["sample"]
    e2e = out["e2e"]
    assert e2e["value"] == out["value"] and e2e["unit"] == out["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_prints_on_rank_zero_only():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3", "--workload",
              "b1h1n256d64", "--gpus", "2"],
             {"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_fewer_than_three_warmup_steps_rejected():
    r = _run(["--warmup", "2"])
    assert r.returncode == 2
