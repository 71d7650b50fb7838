"""Host side of the N-GPU bench on CPU: two gloo ranks shard the sequences with
no overlap and agree on the max-over-ranks step time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        seqs = bench.shard_sequences(16, r)
        gathered = [None] * world
        dist.all_gather_object(gathered, seqs)
        t = bench.max_over_ranks(1.5 + rank, world)
        out[rank] = (gathered, t)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_take_the_max():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        gathered, t = out[rank]
        assert t == pytest.approx(2.5)
        flat = [s for g in gathered for s in g]
        assert sorted(flat) == list(range(32)) and len(set(flat)) == 32
