"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): the
slowest rank's time is what every rank reports, the whole-job throughput adds
every rank's work, and the oracle arm runs on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank
    got = bench.max_over_ranks(ms, world, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_aggregate_is_whole_job():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.aggregate_tflops(1e12, 1, 1.0)
    assert abs(one - 1000.0) < 1e-9
    assert abs(bench.aggregate_tflops(1e12, 4, 1.0) - 4000.0) < 1e-9


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from exact_tiled_attention_22_gb300.inputs import WORKLOADS
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 5, 3, 2

    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.reference_arm(A, WORKLOADS["long"]) == 0
    assert buf.getvalue() == ""

