"""bench.py's reference arm (the fp64 oracle on the host cores) keeps the
JSON-line contract: one line from rank 0 only, with the GPU arm's metric,
unit and workload, a cpu_baseline describing the run, and an e2e object.
Runs on CPU on the base-shape layer (a fraction of a second per step)."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


def _lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check(line, n_gpus):
    assert KEYS <= set(line)
    assert line["impl"] == "reference"
    assert line["metric"] == "MHA layer tokens/s" and line["unit"] == "tokens/s"
    assert line["n_gpus"] == n_gpus and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("mha self-attention base shape")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "1",
                        "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = _lines(r.stdout)
    assert len(lines) == 1
    _check(lines[0], 1)


def test_reference_arm_two_ranks_prints_once():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--workload", "1", "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = _lines(r.stdout)
    assert len(lines) == 1
    _check(lines[0], 2)


def test_reference_arm_attention_workload_config_matches_gpu_arm():
    """On an attention workload the reference arm's config is the object the
    GPU arm prints (mask, flops, L2 treatment included)."""
    import bench
    from transformer_head_scaled_03_gb300.inputs import WORKLOADS, sdpa_inputs
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "2",
                        "--steps", "1", "--warmup", "3", "--cpu-rows-per-head", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = _lines(r.stdout)
    assert len(lines) == 1
    w = WORKLOADS[2]
    assert lines[0]["config"] == json.loads(json.dumps(bench.sdpa_config(w, sdpa_inputs(w)[3], 1)))
    assert lines[0]["unit"] == "TFLOP/s" and lines[0]["value"] > 0
