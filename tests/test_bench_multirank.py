"""The bench's N > 1 host logic on CPU, with world_size-2 gloo process groups.

Under torchrun every rank runs its own GEMM (replicas: weak scaling, no
data-path collective); the timed-region times are reduced with a maximum over
ranks, and the job's value is the work of all ranks over the slowest rank's
time. The reference arm runs on rank 0 only. No GPU is used here: the ranks
are plain processes on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO_ROOT"])
import torch.distributed as dist
import bench
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo", rank=rank, world_size=world)
local = [1.0 + 2.0 * rank, 10.0 - rank, 5.0]
mx = bench.max_over_ranks(local, world)
dist.barrier()
value = bench.job_throughput(world, 10, 1e12, mx[0], 1e12)
dist.destroy_process_group()
print(json.dumps({"rank": rank, "max": mx, "value": value}))
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, world: int, port: int) -> dict:
    env = dict(os.environ)
    env.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank), "MASTER_ADDR": "127.0.0.1",
                "MASTER_PORT": str(port), "REPO_ROOT": ROOT, "CUDA_VISIBLE_DEVICES": ""})
    return env


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], env=_env(r, 2, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        # element-wise maximum of rank 0's [1, 10, 5] and rank 1's [3, 9, 5]
        assert o["max"] == [3.0, 10.0, 5.0]
        # 2 ranks x 10 steps x 1e12 flops over the slowest 3 ms
        assert o["value"] == pytest.approx(2 * 10 * 1e12 / 3e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([2.5, 1.0], 1) == [2.5, 1.0]
    assert bench.job_throughput(1, 4, 2e9, 8.0, 1e9) == pytest.approx(1000.0)


def _bench(args, env, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env, cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_runs_on_rank_zero_only():
    # rank 1 of 2 exits 0 without work and prints nothing
    r = _bench(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny"],
               _env(1, 2, _free_port()))
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_prints_one_contract_line():
    r = _bench(["--impl", "reference", "--steps", "2", "--warmup", "1", "--workload", "tiny"],
               _env(0, 1, _free_port()))
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_gpus_without_torchrun_is_refused():
    env = _env(0, 1, _free_port())
    r = _bench(["--gpus", "2", "--steps", "1", "--warmup", "0"], env)
    assert r.returncode != 0
    assert "torchrun" in (r.stderr + r.stdout)
