"""The reference arm of bench.py (the CPU oracle timed on a bounded sample of the step):
its JSON line keeps the bench contract, and under torchrun only rank 0 runs and prints.
CPU only; the tiny workload keeps each run to a second or two."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "2", "--warmup", "1"]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_line_keeps_the_contract():
    r = _run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["unit"] == "steps/s" and d["higher_is_better"] is True and d["value"] > 0
    # steps x ms_per_step is the time actually spent on samples; the rate is their stated scaling
    ex = d["extrapolated"]
    assert ex["ms_per_sample"] == d["ms_per_step"]
    assert abs(ex["ms_per_full_step"] - 1e3 / d["value"]) <= 1e-3 * ex["ms_per_full_step"] + 0.01
    assert abs(ex["scale"] - ex["ms_per_full_step"] / ex["ms_per_sample"]) <= 1e-2 * ex["scale"]
    # the GPU arm's config dict
    assert d["config"] == bench.config_dict(bench.synth.WORKLOADS["tiny"], 32, 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "2 of 2 sequences" in cb["sample"]                 # the sample never exceeds the batch
    assert d["e2e"] == {"value": d["value"], "unit": "steps/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["gpu_launches"] == 0 and d["vs_baseline"] is None


def test_reference_non_zero_rank_exits_quietly():
    r = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
