"""Host logic of the multi-GPU (weak-scaling replica) bench path, on CPU with
two gloo ranks: each rank gets its own shard, and the timing reduction is the
max over ranks while the work is summed."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, local = bench.dist_env()
    wl = bench.rank_workload(r)
    t = bench.reduce_max(1.0 + r, w)
    f = bench.reduce_sum(10.0 * (r + 1), w)
    bench.barrier(w)
    out[rank] = (r, w, local, wl.seed, wl.batch, wl.total_q, t, f)
    dist.destroy_process_group()


def test_two_rank_shards_and_reductions():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:   # no fork of a multi-threaded process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    (r0, w0, l0, s0, b0, t0, mx0, sm0), (r1, w1, l1, s1, b1, t1, mx1, sm1) = res[0], res[1]
    assert (r0, r1, w0, w1) == (0, 1, 2, 2)
    assert s0 != s1 and b0 == b1 == 64          # same shape, own shard
    assert mx0 == mx1 == 2.0                     # time: max over ranks
    assert sm0 == sm1 == 30.0                    # work: summed over ranks
