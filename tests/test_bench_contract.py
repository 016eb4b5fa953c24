"""bench.py's command line and the JSON line of its reference arm (the oracle timed on host cores).

The reference arm runs on CPU, so its line is checked here in full; the GPU arm's line has the same
keys plus roofline, gpu_launches, clocks and components, and is produced on a GPU machine.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       cwd=ROOT, env=env, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    return p.stdout


def test_defaults_match_the_contract():
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse_args([])
    assert (a.gpus, a.impl, a.warmup >= 3, a.steps >= 1) == (1, "ours", True, True)
    assert a.workload == "model7b" and a.rank is None and a.streams is None
    from rank_gradient_sketching_02_gb300 import synth
    assert synth.WORKLOADS[a.workload].r == 256          # the rank of the 7B-class configuration


def test_reference_arm_prints_one_complete_line():
    out = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0",
                "--cpu-seconds", "0.2"])
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["config"]["workload"] == "tiny"
    sys.path.insert(0, ROOT)
    import bench
    from rank_gradient_sketching_02_gb300 import synth
    w = synth.WORKLOADS["tiny"]
    # the same config object as the GPU arm builds for this workload
    assert d["config"] == bench.workload_config(w, w.layers, w.microbatches, w.r, 1, 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert (e["value"], e["unit"], e["h2d_bytes_per_step"], e["d2h_bytes_per_step"]) == (d["value"], "TFLOP/s", 0, 0)


def test_reference_arm_other_ranks_exit_quietly():
    out = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0"], {"RANK": "1"})
    assert out.strip() == ""
