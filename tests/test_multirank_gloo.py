"""Multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

Every workload is a batch of independent transforms, so N GPUs run N replicas with no
collective on the data path (weak scaling); what crosses ranks is only the start/stop barrier
and the max-over-ranks step time.  These tests run that logic as two spawned processes on the
gloo backend.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="CPU test of the gloo path (with CUDA present the bench picks NCCL)")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench

    w_, r_, _, pg = bench.dist_init(None)
    step = bench.max_over_ranks(pg, 1.0 + rank)  # rank 1 is the slow one
    bench.barrier(pg)
    wl = bench.Workload.with_rows("c2c_1024", 8)
    x = bench.make_inputs(wl, 1 + r_)  # each rank draws its own seeded batch
    gflops, _ = bench.job_rates(wl, w_, step)
    q.put((r_, w_, step, float(abs(x).sum()), gflops, wl.flops))
    pg.destroy_process_group()


def test_two_gloo_ranks_share_the_step_time_not_the_data():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs)
    assert [r[0] for r in res] == [0, 1] and [r[1] for r in res] == [2, 2]
    assert [r[2] for r in res] == [2.0, 2.0]  # max over ranks
    assert res[0][3] != res[1][3]  # different seeded inputs per rank
    # whole-job rate: both ranks' work over the slowest rank's step time
    assert res[0][4] == pytest.approx(2 * res[0][5] / 2e-3 / 1e9)


def test_single_process_has_no_group():
    import bench

    os.environ.pop("WORLD_SIZE", None)
    world, rank, local, pg = bench.dist_init(None)
    assert (world, rank, local, pg) == (1, 0, 0, None)
    assert bench.max_over_ranks(None, 3.5) == 3.5
