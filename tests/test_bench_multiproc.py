"""Host logic of the multi-GPU bench on CPU: two gloo ranks on 127.0.0.1.

Each rank verifies its own batch (weak scaling, no data-path collective); the only exchange is
the timing reduction.  These tests check that reduction, the barrier, the per-rank seeds and
the whole-job rate with world_size 2, without a GPU.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.rank_env()
        bench.barrier(w)
        ms = 2.0 + 3.0 * r                     # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, w)
        rate = bench.whole_job_rate(1.0, w, ms_max)
        seed = bench.rank_seed(4, r)
        wl = bench.workload(r, batch=8)
        out.put((r, w, lr, ms_max, rate, seed, wl.seed, wl.B))
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_reduce_timing_and_seed_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(240)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    (r0, w0, l0, m0, v0, s0, ws0, b0), (r1, w1, l1, m1, v1, s1, ws1, b1) = res
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert m0 == m1 == 5.0                       # max over ranks
    assert v0 == v1 == pytest.approx(2 * 1000.0 / 5.0)   # both ranks' rounds over the slowest time
    assert s0 != s1 and ws0 != ws1                  # each rank draws its own batch
    assert b0 == b1 == 8


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.whole_job_rate(1.0, 1, 0.5) == pytest.approx(2000.0)
    assert bench.rank_seed(4, 0) == 4


def test_stats_traffic_from_committed_capture():
    """The bench's roofline traffic comes from the committed ncu summary only while the
    statistics pass's sources are unchanged; it must then be close to the algorithmic bytes."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.stats_traffic(128) is None
    t = bench.stats_traffic(512)
    if t is not None:
        alg = (512 * 6 + 256 * 5) * 128256 * 2
        assert alg <= t < 1.02 * alg
