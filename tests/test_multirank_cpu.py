"""The multi-rank host logic on CPU with two gloo ranks: head sharding covers
every (batch, head) exactly once, sharded oracle results gathered across
ranks equal the unsharded ones (heads are independent -- no exchange step),
and the benchmark's timing reduction takes the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q, k, v, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        b, h, sq, d = q.shape
        bh = b * h
        lo, hi = bench.shard_heads(bh, world, rank)
        qf, kf, vf = (t.reshape(bh, 1, t.shape[2], d)[lo:hi] for t in (q, k, v))
        o, lse = oracle.attn_fwd(qf.numpy()[None, :, 0], kf.numpy()[None, :, 0], vf.numpy()[None, :, 0], True, 0.3)
        parts = [None] * world
        dist.all_gather_object(parts, (lo, hi, o, lse))
        slowest = bench.max_over_ranks(10.0 + rank, dist, torch.device("cpu"))
        if rank == 0:
            np.save(os.path.join(out_dir, "slowest.npy"), np.array([slowest]))
            o_all = np.concatenate([p[2][0] for p in parts], axis=0)
            l_all = np.concatenate([p[3][0] for p in parts], axis=0)
            np.save(os.path.join(out_dir, "o.npy"), o_all)
            np.save(os.path.join(out_dir, "lse.npy"), l_all)
            np.save(os.path.join(out_dir, "ranges.npy"), np.array([(p[0], p[1]) for p in parts]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("bh,world", [(7, 2), (1, 2), (64, 3), (5, 5)])
def test_shard_heads_partitions(bh, world):
    ranges = [bench.shard_heads(bh, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == bh
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_match_unsharded(tmp_path):
    import oracle
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, 5, 33, 16, generator=g, dtype=torch.float64)
    k = torch.randn(1, 5, 33, 16, generator=g, dtype=torch.float64)
    v = torch.randn(1, 5, 33, 16, generator=g, dtype=torch.float64)
    mp.start_processes(_worker, args=(2, _free_port(), q, k, v, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    o_ref, lse_ref = oracle.attn_fwd(q.numpy(), k.numpy(), v.numpy(), True, 0.3)
    o = np.load(tmp_path / "o.npy")
    lse = np.load(tmp_path / "lse.npy")
    assert np.array_equal(o, o_ref[0]) and np.array_equal(lse, lse_ref[0])
    assert np.load(tmp_path / "ranges.npy").tolist() == [[0, 3], [3, 5]]
    assert float(np.load(tmp_path / "slowest.npy")[0]) == 11.0
