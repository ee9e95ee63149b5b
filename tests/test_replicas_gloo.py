"""The multi-GPU benchmark runs one independent replica per rank (the path
needs no exchange: each rank holds a whole compressed matrix).  Its host
logic -- the slowest rank's time and the throughput of all replicas -- is
checked here with two gloo ranks on the CPU."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_path):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.5, 20.0][rank]                     # rank 1 is the slow one
    slowest = bench.max_over_ranks(torch, dist, ms, "cpu")
    value = bench.replica_throughput(80_000_000, 100, world, slowest)
    gathered = [None] * world
    dist.all_gather_object(gathered, {"rank": rank, "slowest": slowest, "value": value})
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump(gathered, f)
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank(tmp_path):
    out = tmp_path / "ranks.json"
    mp.start_processes(_rank, args=(2, _free_port(), str(out)), nprocs=2, start_method="spawn", join=True)
    ranks = json.loads(out.read_text())
    assert [r["slowest"] for r in ranks] == [20.0, 20.0]
    # 2 replicas x 100 steps x 80 MB in 20 ms
    assert all(r["value"] == pytest.approx(2 * 100 * 80e6 / 0.020 / 1e9) for r in ranks)
