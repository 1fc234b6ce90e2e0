"""bench.py's multi-process plumbing on CPU: world size 2 over gloo.

The path shards into independent per-rank problems (no data-path collective):
each rank times its own shard, the ranks meet at a barrier on both sides of
the timed region, and the reported time is the maximum over ranks.  This
checks that plumbing (rendezvous on 127.0.0.1, barrier, max-over-ranks) and
the per-rank seeding of the shards without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
from tiled_attention_flashattention_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # each rank reports a different "elapsed time"; everyone must see the max
    t = bench.max_over_ranks(1.5 + rank, w)
    # per-rank shards are seeded differently (independent problems)
    c = wl.WORKLOADS["mha_b1_h2_n128_d64"]
    shard = wl.PrefillCase(**{**c.__dict__, "seed": c.seed + 1000 * r})
    q = wl.prefill_inputs(shard)[0].float()
    out[rank] = (t, float(q.sum()))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_gloo_barrier_and_max():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 2.5
    assert out[0][1] != out[1][1]          # different shards


def test_gpus_flag_must_match_world_size(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    with pytest.raises(SystemExit):
        bench.dist_setup(2)
