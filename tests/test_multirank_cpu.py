"""Multi-rank host logic of bench.py on the CPU (gloo, world size 2).

The decode path runs one independent problem per rank; the only cross-rank
steps are the barrier and the max-over-ranks of every measured time.  These
tests run that logic on two CPU processes, and check that the reference arm
under a multi-rank launch runs on rank 0 only.
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
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 1.5 + 2.0 * rank                      # each rank measured something different
        results[rank] = bench._max_over_ranks(mine, world, torch.device("cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), results), nprocs=2,
                           start_method="spawn")
        assert dict(results) == {0: 3.5, 1: 3.5}


def test_single_rank_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(2.25, 1, torch.device("cpu")) == 2.25


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank0_only(rank):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 0:
        assert len(lines) == 1
        rec = json.loads(lines[0])
        assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
        assert rec["cpu_baseline"]["kind"] == "oracle"
        assert rec["e2e"]["h2d_bytes_per_step"] == 0
    else:
        assert lines == []
