"""The multi-GPU story of this path is replicas (each rank runs the whole
workload; output channels would shard, but the pages have no exchange step):
bench.py takes the slowest rank's time and reports the whole-job throughput.
Checked here with two gloo ranks on the CPU -- no GPU, no NCCL."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.max_over_ranks(times[rank], world)
        w = bench.WORKLOADS["w4a16_gemv_m1"]
        value, unit = bench.metric_of(w, ms, world)
        out.put((rank, ms, value, unit))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(3.5, 4.25), (7.0, 1.0)])
def test_two_replicas_take_the_slowest_rank(times):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    sys.path.insert(0, ROOT)
    import bench
    w = bench.WORKLOADS["w4a16_gemv_m1"]
    slow = max(times)
    for rank, ms, value, unit in res:
        assert ms == slow                                   # every rank sees the max
        one, _ = bench.metric_of(w, slow, 1)
        assert value == pytest.approx(2 * one)              # whole-job value = 2 replicas' work in the slow time
        assert unit == "GB/s"


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.replica_value(10.0, 2.0, 4) == 20.0
