"""The benchmark's multi-rank bookkeeping on CPU with the gloo backend (world size 2): the
timing reduction takes the slowest rank, and whole-job throughput counts every rank's work.
Ranks run independent replicas, so there is no data-path collective to test."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, lr = bench.dist_info()
    assert (ws, r, lr) == (world, rank, rank)
    t_local = 1.0 + rank  # rank 1 is slower
    t_max = bench.max_over_ranks(t_local, world)
    bench.barrier(world)
    out[rank] = t_max
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 2.0, 1: 2.0}


def test_single_rank_is_identity(monkeypatch):
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.dist_info()[0] == 1
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_algorithmic_bytes_counts_prefix_once():
    import bench
    import workloads as W
    wl = W.llama8b_single_prefix_16k(0)
    s = wl.spec
    lens = [wl.cold_len(b) for b in range(s.B)]
    one = bench.algorithmic_bytes(s, [0] * s.B, lens, 2)
    row = s.n_kv * s.d * 2
    assert one == 2 * 16384 * row + sum(2 * L * row + 4 * L for L in lens) + 2 * s.B * s.n_q * s.d * 2 + 4 * s.B * s.n_q
    # flops count the prefix per request (every query still attends over it)
    f = bench.algorithmic_flops(s, [0] * s.B, lens)
    assert f == 4 * s.d * s.n_q * sum(16384 + L for L in lens)
