"""The multi-rank host logic on CPU with a world-size-2 gloo group: sequences are sharded
across ranks with no collective on the data path, the sharded results equal the unsharded
ones, and the benchmark's whole-job figure uses the slowest rank's time."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank decodes its own sequences of one shared batch
        x = W.make_gqa(5, 8, 2, 16, [3, 40, 17, 64, 9], page_size=8, shuffle=True, seed=3,
                       dtype=torch.float32)
        lo, hi = bench.shard_range(x.B, rank, world)
        out, _ = oracle.gqa(x.q[lo:hi], x.k_pool, x.v_pool, x.block_table[lo:hi],
                            x.seq_lens[lo:hi], x.scale)
        np.save(os.path.join(out_dir, f"shard{rank}.npy"), out)
        # whole-job throughput over the slowest rank
        ms, gbs = bench.aggregate(10.0 + 5.0 * rank, 1e9, world, dist)
        np.save(os.path.join(out_dir, f"agg{rank}.npy"), np.array([ms, gbs]))
    finally:
        dist.destroy_process_group()


def test_shard_range_covers_everything():
    for n in (1, 2, 5, 32, 33):
        for world in (1, 2, 3, 8):
            parts = [bench.shard_range(n, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(parts[i][1] == parts[i + 1][0] for i in range(world - 1))
            assert max(b - a for a, b in parts) - min(b - a for a, b in parts) <= 1


def test_two_rank_gloo_sharding_and_aggregate(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    x = W.make_gqa(5, 8, 2, 16, [3, 40, 17, 64, 9], page_size=8, shuffle=True, seed=3,
                   dtype=torch.float32)
    full, _ = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    got = np.concatenate([np.load(tmp_path / "shard0.npy"), np.load(tmp_path / "shard1.npy")])
    assert np.array_equal(got, full)
    for r in range(2):
        ms, gbs = np.load(tmp_path / f"agg{r}.npy")
        assert ms == 15.0                       # the slowest rank's time
        assert abs(gbs - 2 * 1e9 / 15e-3 / 1e9) < 1e-9
