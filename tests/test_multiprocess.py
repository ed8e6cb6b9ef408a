"""World-size-2 gloo run of the multi-rank logic on CPU: every rank works on
its own shard (independent sequences -- no data-path collective), the timing
is the max over ranks, the rate is whole-job."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import se_workloads as W
    from oracle import cache as ocache
    from oracle import pipelines as opipe
    # each rank: its own shard of sequences (different seeds), no exchange
    shape = W.snapkv_tiny(name=f"snapkv_tiny_rank{rank}")
    inp = W.snapkv_inputs(shape, "cpu")
    c = ocache.from_tensors(inp["cache"])
    r = opipe.snapkv(c, inp["q_win"], inp["q_pos"].numpy(), inp["q_dec"], shape)
    kept = int(c.ctx_len[0])
    ms = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")
    rate = bench.whole_job_rate(shape.ctx, world, ms)
    out[rank] = (kept, ms, rate, float(r["scores"][(0, 0)].sum()))
    dist.destroy_process_group()


def test_two_rank_gloo_replicas():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 128                 # both shards compressed to budget
    assert res[0][1] == res[1][1] == 20.0                # max over ranks
    assert res[0][2] == pytest.approx(512 * 2 / 0.020)   # whole-job rate
    assert res[0][3] != res[1][3]                        # different data per rank
    # each shard's score total is w * G (rows sum to one; here the scored
    # prefix holds most of the mass, the window keys the rest)
    assert 0 < res[0][3] < 32 * 4
