"""The N > 1 path of the benchmark: independent replicas whose timing is the
slowest rank's, aggregated with one all-reduce.  Run here with two gloo ranks
on the CPU (no GPU, no data-path collective)."""
import importlib.util
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    ms = [12.5, 20.0][rank]                   # rank 1 is the slow replica
    slow = b.slowest_rank_ms(ms, world)
    value = b.replica_throughput(8192, 10, world, slow)
    q.put((rank, slow, value))
    dist.destroy_process_group()


def test_two_gloo_replicas_report_the_slowest_rank():
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
    for rank, slow, value in out:
        assert slow == 20.0                      # max over ranks on every rank
        assert value == pytest.approx(2 * 8192 * 10 / 0.020)


def test_single_process_is_a_no_op():
    b = _bench()
    assert b.slowest_rank_ms(7.0, 1) == 7.0
    assert b.replica_throughput(64, 5, 1, 10.0) == pytest.approx(64 * 5 / 0.010)
