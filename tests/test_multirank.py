"""The benchmark's several-GPU logic on CPU ranks (gloo, world size 2): each rank gets its own
shard of inputs, only the step time crosses ranks (a max), and the reported value counts the
work of every rank."""
import os
import socket

import numpy as np
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
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import fa_inputs

        w = fa_inputs.BY_NAME["tiny_gqa_d64"]
        inp = bench.shard_inputs(w, rank)
        local_ms = 10.0 + 5.0 * rank
        m = bench.reduce_max(local_ms, world)
        digest = float(np.asarray(inp.q, np.float64).sum())
        t = torch.tensor([digest], dtype=torch.float64)
        gathered = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(gathered, t)
        out[rank] = (m, [float(g.item()) for g in gathered], inp.q.shape)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(out)
    # the max over ranks is seen by every rank
    assert res[0][0] == res[1][0] == 15.0
    # shards are distinct draws of the same shape
    digests = res[0][1]
    assert digests[0] != digests[1]
    assert res[0][2] == res[1][2]


def test_single_rank_reduce_is_identity():
    import bench

    assert bench.reduce_max(3.5, 1) == 3.5
