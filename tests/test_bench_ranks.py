"""The multi-rank path of bench.py on CPU: two gloo ranks, barrier, max over ranks and the
whole-job (weak-scaling) throughput of independent replicas."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup(0)                 # gpus = 0 -> gloo
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    ms = 10.0 + 5.0 * rank                             # rank 1 is the slow one
    ms_max = bench.max_over_ranks(ms, w)
    out[rank] = (ms_max, bench.replica_throughput(1000.0, ms_max, w))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms_max, rate = out[r]
        assert ms_max == 15.0
        assert abs(rate - 2 * 1000.0 / 0.015) < 1e-6


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_throughput(10.0, 1000.0, 1) == 10.0
