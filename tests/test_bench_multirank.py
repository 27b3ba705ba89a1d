"""bench.py under torchrun on CPU.

The verification path runs on one GPU and has no multi-GPU arm: with more
than one rank the GPU arm must print one "unavailable" line and launch
nothing, and the reference arm (the oracle on the host cores) runs on rank 0
alone while the other ranks exit without work.  No GPU is involved.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(*bench_args, timeout=600):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", *bench_args]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout, env=env)


def json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_gpu_arm_refuses_more_than_one_rank():
    r = torchrun("--gpus", "2", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1
    assert "unavailable" in lines[0] and lines[0]["n_gpus"] == 2
    assert "value" not in lines[0]


def test_gpu_arm_refuses_gpus_flag_without_torchrun():
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "4", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1 and "unavailable" in lines[0]


def test_reference_arm_under_torchrun_prints_one_line():
    r = torchrun("--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
                 "--cpu-budget-s", "0.3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the step time is extrapolated from a bounded sample, and says so
    assert d["ms_per_step_kind"].startswith("extrapolated")
    assert 0 < d["sampled_s_per_step"] < d["ms_per_step"] * 1e-3
