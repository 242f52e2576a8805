"""Replica (data-parallel) host logic of bench.py on CPU with gloo, world
size 2: every rank draws its own independent batch, the per-rank step times
are reduced with MAX, and request shards of a global batch cover it exactly
once."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import gen


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = bench.replica_inputs("tiny", rank)
        digest = float(inp.q.float().sum())
        t = bench.max_over_ranks([1.0 + rank, 10.0 - rank], torch.device("cpu"))
        got = torch.tensor([digest] + t, dtype=torch.float64)
        gathered = [torch.zeros_like(got) for _ in range(world)]
        dist.all_gather(gathered, got)
        if rank == 0:
            torch.save(gathered, out_path)
    finally:
        dist.destroy_process_group()


def test_two_replicas_with_gloo(tmp_path):
    out = str(tmp_path / "res.pt")
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    g = torch.load(out)
    assert g[0][0] != g[1][0]                       # independent batches per replica
    for r in range(2):
        assert g[r][1].item() == 2.0 and g[r][2].item() == 10.0   # MAX over ranks, elementwise


@pytest.mark.parametrize("batch,world", [(64, 1), (64, 2), (7, 3), (5, 8)])
def test_request_shards_cover_the_batch_once(batch, world):
    seen = []
    for r in range(world):
        seen.extend(gen.shard_requests(batch, r, world))
    assert sorted(seen) == list(range(batch))
