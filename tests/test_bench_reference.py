"""bench.py's reference arm (the oracle on the host cores) on the CPU: the one
JSON line and its keys, alone and under torchrun with two ranks, where rank 0
alone prints and every rank exits 0."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--workload", "tiny_fp32", "--steps", "2", "--warmup", "3", "--ref-episodes", "1"]


def _lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check(line, n_gpus):
    assert line["impl"] == "reference" and line["n_gpus"] == n_gpus
    assert line["value"] > 0 and line["unit"] == "tuples/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] >= 3 and line["data"] == "synthetic"
    # the same config object as the GPU arm's line for this workload
    sys.path.insert(0, ROOT)
    import bench
    from rl_experience_collection_gb300 import workloads as wl
    w = wl.WORKLOADS["tiny_fp32"]
    assert line["config"] == bench.workload_config(w, w.n_episodes, w.horizon, n_gpus)
    assert line["config"]["workload"] == "tiny_fp32"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == os.cpu_count() and cb["value"] == line["value"] and cb["sample"]
    assert cb["nproc"] == os.cpu_count() and cb["cpu_model"]
    assert line["e2e"] == {"value": line["value"], "unit": "tuples/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_prints_one_line():
    p = subprocess.run([sys.executable, "bench.py", *ARGS], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _lines(p.stdout)
    assert len(lines) == 1
    _check(lines[0], 1)


def test_reference_arm_under_torchrun_two_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2", *ARGS]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _lines(p.stdout)
    assert len(lines) == 1
    _check(lines[0], 2)
