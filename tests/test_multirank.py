"""The benchmark's multi-rank path on CPU: one process per rank over gloo (world size
2), the barrier, the slowest rank's time, and the summed tokens.  Requests shard
across ranks with no exchange (independent replicas), so this is all the
cross-rank logic there is."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    ws, r, local = bench.dist_setup()
    bench.barrier(ws)
    ms = 10.0 * (r + 1)                       # rank 1 is the slower one
    t_max = bench.max_over_ranks(ms, ws)
    tokens = bench.sum_over_ranks(32 * 5, ws)  # 32 requests x 5 steps per replica
    out[r] = (ws, t_max, tokens, tokens / (t_max / 1e3))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_benchmark():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert sorted(out.keys()) == [0, 1]
    for r in range(world):
        ws, t_max, tokens, value = out[r]
        assert ws == 2 and t_max == 20.0 and tokens == 320.0
        assert value == pytest.approx(320 / 0.020)
