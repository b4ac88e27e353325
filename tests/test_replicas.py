"""The replica path of bench.py (one process per GPU, max-over-ranks timing)
on CPU: two gloo ranks on 127.0.0.1 report different times and both must see
the maximum; the per-layer job time divides by the number of replicas."""
import importlib.util
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        assert b._dist_env() == (world, rank, rank)
        got = b.job_ms(10.0 + 5.0 * rank, world, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_job_time_per_layer_counts_every_replica():
    b = _bench()
    assert b.job_us_per_layer(0.55, 11, 1) == pytest.approx(50.0)
    assert b.job_us_per_layer(0.55, 11, 4) == pytest.approx(12.5)
    assert b.job_ms(3.5, 1, "cpu") == 3.5
