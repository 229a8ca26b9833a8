"""bench.py's reference arm (the oracle timed on the host cores) on the CPU: the JSON line
the benchmark contract asks for, and the silent exit of ranks other than 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_l2", "--steps", "2", "--warmup", "1",
        "--ref-sample-tokens", "16"]


def _run(env_extra=None, extra_args=()):
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env.update(env_extra or {})
    return subprocess.run(ARGS + list(extra_args), capture_output=True, text=True, cwd=ROOT, timeout=600, env=env)


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
    out = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, ["--gpus", "2"])
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_gpus_flag_must_match_the_launched_ranks():
    """A --gpus count that disagrees with the ranks torchrun started is refused, on both arms,
    before any work."""
    for impl in ("reference", "ours"):
        env = {"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"}
        out = subprocess.run([sys.executable, "bench.py", "--impl", impl, "--gpus", "1"], capture_output=True,
                             text=True, cwd=ROOT, timeout=600,
                             env={**{k: v for k, v in os.environ.items()}, **env})
        assert out.returncode == 2, (impl, out.returncode, out.stderr[-2000:])
        assert "does not match WORLD_SIZE" in out.stderr and out.stdout.strip() == ""


def test_gpus_flag_without_torchrun_launches_that_many_ranks():
    """bench.py --gpus 2 run directly starts two ranks itself; rank 0 alone prints the line,
    and it reports the two GPUs (the reference arm needs no GPU, so this runs on the CPU)."""
    out = _run(None, ["--gpus", "2"])
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_l2_note_of_the_timed_workloads():
    sys.path.insert(0, ROOT)
    import bench
    import synth
    for name in ("llama8b_l16", "qwen14b_l24_g4", "llama70b_l40"):
        assert bench.l2_note(synth.WORKLOADS[name].shape).startswith("inputs larger than L2")


def test_step_roofline_arithmetic():
    """Sum over classes of max(FLOPs / peak, bytes / bandwidth), per step, against the step."""
    sys.path.insert(0, ROOT)
    import bench
    prof = {  # totals over 2 steps
        "gemm": {"flops": 2 * 1.0e12, "bytes": 2 * 1.0e9, "ms": 2.4, "calls": 2, "kernels": 2},    # 1.0 ms vs 0.1 ms
        "norm": {"flops": 0.0, "bytes": 2 * 5.0e9, "ms": 1.2, "calls": 2, "kernels": 2},           # 0.5 ms
        "plan": {"flops": 0.0, "bytes": 0.0, "ms": 0.1, "calls": 2, "kernels": 2},                 # 0
    }
    r = bench.step_roofline(prof, steps=2, ms_per_step=2.0, peak_tflops=1000.0, hbm_gbs=10000.0)
    assert abs(r["per_class_ms"]["gemm"] - 1.0) < 1e-12
    assert abs(r["per_class_ms"]["norm"] - 0.5) < 1e-12
    assert r["per_class_ms"]["plan"] == 0.0
    assert abs(r["t_roofline_ms"] - 1.5) < 1e-12 and abs(r["frac"] - 0.75) < 1e-12
    assert list(r["per_class_ms"]) == ["gemm", "norm", "plan"]
