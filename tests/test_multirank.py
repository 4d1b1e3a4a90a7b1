"""The multi-rank (replica) logic of the benchmark on CPU: world size 2 over gloo.

Each rank runs its own copy of the workload (independent heads, no data-path
collective); the ranks only agree on timing.  These tests cover that host-side
logic without a GPU: the process group comes up from the launcher's environment,
the job time is the maximum over ranks, the job value counts every rank's tokens,
and the reference arm runs on rank 0 alone.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local, dist = bench.dist_setup(world)
    ms = 2.0 if rank == 1 else 1.0            # rank 1 is the slow one
    bench.barrier(dist)
    m = bench.allmax(dist, ms)
    q.put((r, w, local, m, bench.job_value(1000, w, m)))
    dist.destroy_process_group()


def _ref_worker(rank, q):
    # the reference arm on a non-zero rank returns at once, without work or output
    os.environ.update(RANK=str(rank), WORLD_SIZE="2")
    sys.path.insert(0, ROOT)
    import bench

    class A:
        gpus, steps, warmup = 2, 1, 0
    q.put((rank, bench.run_reference(A, None)))


def _run(target, args_list):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=target, args=a + (q,)) for a in args_list]
    for p in ps:
        p.start()
    out = [q.get(timeout=120) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_two_rank_timing_takes_the_slowest_rank():
    port = _free_port()
    res = _run(_worker, [(0, 2, port), (1, 2, port)])
    assert [r[0] for r in res] == [0, 1]
    for rank, world, local, m, value in res:
        assert world == 2 and local == rank
        assert m == 2.0                          # max over ranks
        assert value == pytest.approx(1000 * 2 / 2e-3)


def test_reference_arm_idles_on_other_ranks():
    res = _run(_ref_worker, [(1,)])
    assert res == [(1, 0)]
