"""Multi-rank arithmetic of bench.py on CPU (gloo, world size 2): each rank
runs its own replica; the reported time is the slowest rank's and the rate
counts every rank's sequences.  No GPU is involved."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        dist.barrier()
        m = bench.max_over_ranks(times[rank], world)
        v = bench.aggregate_rate(world, 256, 10, m)
        out[rank] = (m, v)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rate_gloo():
    world = 2
    times = [12.5, 20.0]
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
    for r in range(world):
        m, v = out[r]
        assert m == pytest.approx(20.0)
        assert v == pytest.approx(2 * 256 * 10 / 20e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_rate(1, 256, 4, 2.0) == pytest.approx(256 * 4 / 2e-3)


def test_shared_prefix_unique_bytes_counts_each_tile_once():
    """The shared-prefix line's unique bytes equal decode_bytes' total minus
    the K/V of every repeated (physical block, row) that the tables name
    more than once: counted here directly from the block tables."""
    import numpy as np

    import bench
    from paged_kv_cache_151_gb300 import workloads as wl

    b = wl.shared_prefix(batch=12, prefix_blocks=8, lo=5, hi=40, canary=False)
    total = bench.decode_bytes(b)["total"]
    per_tok = 2 * b.num_kv_heads * b.head_dim * 2
    seen, repeats = set(), 0
    for s in range(b.num_seqs):
        for t in range(int(b.seq_lens[s])):
            key = (int(b.block_tables[s, t // 16]), t % 16)
            repeats += key in seen
            seen.add(key)
    assert repeats == (b.num_seqs - 1) * int(b.meta["prefix_tokens"])
    assert bench.shared_prefix_unique_bytes(b) == total - repeats * per_tok
    assert np.all(b.block_tables[:, :8] == b.block_tables[0, :8])
