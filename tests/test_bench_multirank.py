"""The bench's multi-rank bookkeeping on CPU: two gloo ranks agree on the slowest rank's
time and on the whole-job throughput (weak scaling, no collective on the data path)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, lr, w = bench.dist_env()
    t = bench.max_over_ranks(1.0 + rank * 0.5, w)      # rank 1 is the slower one
    v = bench.job_throughput(1e9, 10, w, t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, lr, w, t, v))


def test_two_gloo_ranks_agree():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[2] == 2 for o in out)
    assert all(o[3] == 1.5 for o in out)                 # max over ranks
    assert all(abs(o[4] - 2 * 1e9 * 10 / 1.5 / 1e9) < 1e-9 for o in out)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_throughput(2e9, 5, 1, 2.0) == 5.0
