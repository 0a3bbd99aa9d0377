"""The multi-process path of bench.py on CPU: two gloo ranks (world size 2),
rendezvous on 127.0.0.1.  Each rank reports its own step time; both must see the
maximum, and the whole-job value is world x tokens / max time (weak scaling,
independent replicas, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 2.0 + 3.0 * rank            # rank 1 is the slow one
        ms = bench.reduce_max(local_ms, "cpu")
        out[rank] = (ms, bench.weak_scaling_value(8192, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_weak_scaling_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == pytest.approx(5.0)
    assert value == pytest.approx(2 * 8192 / 5e-3)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.weak_scaling_value(100, 1, 2.0) == pytest.approx(50000.0)
