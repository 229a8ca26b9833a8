"""bench.py's reference arm (the oracle timed on the host cores) on the CPU: the JSON line
the benchmark contract asks for, and the silent exit of ranks other than 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_l2", "--steps", "2", "--warmup", "1",
        "--ref-sample-tokens", "16"]


def _run(env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run(ARGS, capture_output=True, text=True, cwd=ROOT, timeout=600, env=env)


def test_reference_arm_prints_the_contract_line():
    out = _run()
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["unit"] == "tokens/s"
    assert d["config"]["workload"].startswith("tiny_l2")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the tiny shape fits in L2 and says so
    assert "fit in L2" in d["config"]["l2"]


def test_reference_arm_other_ranks_exit_quietly():
    out = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_l2_note_of_the_timed_workloads():
    sys.path.insert(0, ROOT)
    import bench
    import synth
    for name in ("llama8b_l16", "qwen14b_l24_g4", "llama70b_l40"):
        assert bench.l2_note(synth.WORKLOADS[name].shape).startswith("inputs larger than L2")
