"""World-size-2 gloo runs on CPU of the multi-rank host logic (no GPU is touched):

* the exchange step of the DSA top-k producer: rank s plays shard s, its candidate lists
  are all-gathered in shard order by ``dcp_topk_gather`` and merged; the merge of the
  gathered lists must be the top-k of the unsharded scores (LMDeploy PR #4952, Summary:
  DSA merges local candidates into the global top-k).  The lists and the merge come from
  the oracle here; the kernels that produce them on a GPU are checked in test_gpu_topk.py;
* the bench's aggregation over ranks: every rank learns the slowest rank's time and the
  whole-job rate counts the units of all ranks."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, job):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        job(rank, world)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _topk_exchange(rank, world):
    import decode_context_sparse_gb300 as dcp
    from oracle import topk as otk
    D, I, k = world, 1, 64
    rng = np.random.default_rng(5)  # the same global scores on every rank
    row_len = np.array([3000, 2999, 10, 0, 130])
    R = row_len.size
    glob = np.round(rng.standard_normal((R, 3000)) * 4).astype(np.float32) / 4
    n = [oracle.count_owned(int(L), D, I, rank) for L in row_len]
    g = otk.shard_slots(max(n), D, I, rank)
    sc = np.full((1, R, max(n) + 1), np.nan, dtype=np.float32)
    for r in range(R):
        sc[0, r, :n[r]] = glob[r, g[:n[r]]]
    cs, ci = otk.local_topk(sc, np.array([n]), k, D, I, shard=rank)
    gs, gi = dcp.dcp_topk_gather(torch.from_numpy(cs), torch.from_numpy(ci))
    assert tuple(gs.shape) == (D, R, k) and tuple(gi.shape) == (D, R, k)
    assert np.array_equal(gi[rank].numpy(), ci[0])
    assert np.array_equal(gs[rank].numpy().view(np.int32), cs[0].view(np.int32))
    top, cnt = otk.merge_topk(gs.numpy(), gi.numpy(), k)
    want, wcnt = otk.global_topk(glob, row_len, k)
    assert np.array_equal(top, want) and np.array_equal(cnt, wcnt)


def _bench_aggregate(rank, world):
    import bench
    t = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
    assert t == 10.0 + 5.0 * (world - 1)
    rate = bench.whole_job_rate(384, 20, t, world)
    assert abs(rate - world * 384 * 20 / (t / 1e3)) < 1e-6


def _spawn(job, world=2):
    oracle.build()  # compiled once, before the ranks start
    mp.spawn(_worker, args=(world, _free_port(), job), nprocs=world, join=True)


def test_topk_exchange_two_ranks():
    _spawn(_topk_exchange)


def test_bench_aggregation_two_ranks():
    _spawn(_bench_aggregate)
