"""The N > 1 host path of bench.py on CPU ranks (gloo, world size 2).

On several GPUs the layer runs as independent replicas: no collective touches the data,
each rank draws its own token batch, and the job's time is the slowest rank's.  These
tests run that host logic as two gloo processes on 127.0.0.1; no GPU is involved.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import synth

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the slowest rank's time is every rank's result
        own = [3.25, 7.5][rank]
        got = bench.max_over_ranks(own, world, torch.device("cpu"))
        # replicas draw different token batches from the same workload
        shape = synth.WORKLOADS["toy"]
        inp = synth.make_inputs(shape.with_(seed=bench.replica_seed(shape, rank)), device="cpu")
        x_sum = float(inp["x"].double().sum())
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"max": got, "x_sum": x_sum, "T": int(inp["x"].shape[0])}, f)
    finally:
        dist.destroy_process_group()


def test_replicas_max_over_ranks_and_own_batches(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r = [json.load(open(tmp_path / f"r{i}.json")) for i in range(world)]
    assert r[0]["max"] == r[1]["max"] == 7.5
    assert r[0]["T"] == r[1]["T"]
    assert r[0]["x_sum"] != r[1]["x_sum"]


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(2.5, 1, torch.device("cpu")) == 2.5


def test_reference_arm_under_torchrun_prints_one_line():
    """`--impl reference` launched as two ranks: rank 0 alone times the oracle and prints
    one JSON line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--config", "toy", "--steps", "1",
           "--warmup", "1", "--cpu-sample", "4"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["unit"] == "tokens/s" and res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle"
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["d2h_bytes_per_step"] == 0
