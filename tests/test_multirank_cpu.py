"""The N>1 host path of bench.py on CPU ranks (gloo, world size 2): each rank
draws its own batch of the same workload shape (weak scaling, no collective
on the data path) and the job time is the slowest rank's."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from deepseek_top_sparse_gb300 import workloads

    inp = workloads.v4_ratio4_decode(seed=bench.rank_seed(rank), B=4, long_ctx=4096, short_hi=1024)
    job = bench.max_over_ranks(1.0 + 0.5 * rank)
    q.put((rank, job, tuple(inp.q.shape), int(inp.topk_idxs.sum()), float(inp.q.float().sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_weak_scaling_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, job0, shp0, isum0, qsum0), (r1, job1, shp1, isum1, qsum1) = out
    assert job0 == job1 == 1.5            # the slowest rank's time on every rank
    assert shp0 == shp1                   # same per-rank workload shape (weak scaling)
    assert (isum0, qsum0) != (isum1, qsum1)  # but each rank's own batch


def test_single_process_max_is_identity():
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.rank_seed(0) != bench.rank_seed(1)
