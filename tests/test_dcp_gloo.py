"""The multi-rank host logic on the CPU with two gloo ranks: each rank owns
every other KV page of each request (decode-context-parallel layout),
computes its shard's partial result, the ranks exchange (out, lse) with an
all-gather, and the LSE merge equals the unsharded attention. Also checks the
benchmark's max-over-ranks timing reduction. No GPU."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.attention as att
import oracle.merge as merge
from workloads import make_batch_from_lengths, shard_pages


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle(b):
    return att.mla_decode(b.q.numpy(), b.kv.numpy(), b.block_table.numpy(), b.seq_lens.numpy(),
                          b.k, b.sm_scale, b.q_scale, b.kv_scale)


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = make_batch_from_lengths((300, 65, 7), 2, 3, seed=5, scaling="amax")
        o, l = _oracle(shard_pages(b, world, rank))
        o_all = [torch.empty(o.shape, dtype=torch.float64) for _ in range(world)]
        l_all = [torch.empty(l.shape, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(o_all, torch.from_numpy(o))
        dist.all_gather(l_all, torch.from_numpy(l))
        mo, ml = merge.combine(np.stack([t.numpy().reshape(-1, 512) for t in o_all]),
                               np.stack([t.numpy().reshape(-1) for t in l_all]))
        ro, rl = _oracle(b)
        err = max(np.abs(mo - ro.reshape(-1, 512)).max(), np.abs(ml - rl.reshape(-1)).max())
        # the benchmark's reduction: the slowest rank's time sets the value
        import bench
        t = bench.max_over_ranks([1.0 + rank, 10.0 - rank], torch.device("cpu"))
        results[rank] = (float(err), t)
    finally:
        dist.destroy_process_group()


def test_two_rank_exchange_and_merge():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), results), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(results)
    for rank in (0, 1):
        err, t = res[rank]
        assert err < 1e-12
        assert t == [2.0, 10.0]
