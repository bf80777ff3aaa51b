"""bench.py's multi-rank bookkeeping with two ranks on the CPU (gloo).

Every (batch, head) sequence is independent, so N GPUs run N replicas of the
workload with no collective on the data path; the only cross-rank steps are
the barriers around the timed region and the maximum of the ranks' times,
from which the whole-job throughput (units of all ranks / slowest time) is
formed. These run here as two gloo processes on 127.0.0.1.
"""
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    # gloo ranks on the CPU, whether or not this machine has GPUs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), LA_DIST_BACKEND="gloo")
    import sys
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_init()
    try:
        bench.barrier(w)
        slowest = bench.max_over_ranks(times[r], w)
        bench.barrier(w)
        out.put((r, w, local, dist.get_backend(), slowest))
    finally:
        dist.destroy_process_group()


def _run(world, times):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=120) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return res


def test_two_ranks_agree_on_the_slowest_time():
    times = [0.125, 0.5]
    res = _run(2, times)
    assert [r[0] for r in res] == [0, 1]
    for rank, world, local, backend, slowest in res:
        assert world == 2 and local == rank and backend == "gloo"
        assert slowest == max(times)
