"""The multi-rank (replica) path of bench.py, on CPU with gloo at world size 2.

Requests are independent, so N GPUs run N replicas: each rank verifies its own batch (seeded by
its rank), no collective touches the data path, and the job's throughput is the sum over ranks of
the tokens verified per step divided by the slowest rank's step time.  These tests run the same
helpers under a real two-process gloo group, and the reference arm under torchrun.
"""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup(world, backend="gloo")
    try:
        assert (w, r) == (world, rank)
        wl = bench.make_workload("small", r)
        # a fake per-rank step time: the job's time is the slowest rank's
        ms = bench.max_over_ranks(1.0 + r, w)
        bench.barrier(w)
        value = bench.job_throughput(w, wl.B, wl.D, ms)
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump({"ms": ms, "value": value, "B": wl.B, "D": wl.D,
                       "L": [int(x) for x in wl.L], "draft0": wl.draft[0].tolist()}, f)
    finally:
        dist.destroy_process_group()


def test_replica_helpers_under_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    # max over ranks reached every rank
    assert [r["ms"] for r in res] == [2.0, 2.0]
    # whole-job throughput: both ranks' tokens over the slowest step
    want = world * res[0]["B"] * res[0]["D"] / 2e-3
    assert all(r["value"] == pytest.approx(want) for r in res)
    # the ranks verify different requests (seeded by rank), not copies of one batch
    assert res[0]["draft0"] != res[1]["draft0"]


def test_reference_arm_under_torchrun():
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "tiny"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout   # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
