"""Replica bookkeeping of bench.py for N > 1, on CPU with the gloo backend:
every rank runs its own copy of the workload, the timed region is bracketed
by barriers and the reported time is the maximum over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    rk = bench.Ranks(backend="gloo")
    assert (rk.rank, rk.world) == (rank, world)
    rk.barrier()
    ms = 2.0 + rank  # rank r took 2 + r ms per step
    m = rk.max(ms)
    out[rank] = (m, bench.aggregate_tflops(rk.world, 1e12, m))
    rk.barrier()
    rk.close()


def test_two_gloo_ranks_take_max_and_aggregate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for m, v in res.values():
        assert m == pytest.approx(3.0)  # the slowest rank decides
        assert v == pytest.approx(2 * 1e12 / 3e-3 / 1e12)  # both replicas' work over that time


def test_single_process_is_identity():
    import bench

    rk = bench.Ranks()
    if rk.world == 1:
        assert rk.max(1.5) == 1.5
        assert bench.aggregate_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)
    rk.close()
