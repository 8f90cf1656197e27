"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each timing its own
replica, agree on the max over ranks (weak scaling, no data-path collective)."""
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


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.rank_info()
    assert (r, w, lr) == (rank, world, rank)
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_gpu_launch_count_is_positive_for_every_row_set():
    import bench
    for rows in ({"swap"}, {"decode"}, {"topk"}, {"prefill"}, {"swap", "decode", "topk", "prefill"}):
        assert bench.gpu_launch_count(10, rows) > 0
