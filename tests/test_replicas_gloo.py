"""The multi-process path of the benchmark on CPU: world size 2 over gloo.

With N GPUs the benchmark runs N independent replicas of the layer (each on
its own batch; no collective on the data path) and reports the whole job's
tokens/s over the slowest rank's time.  These tests run that aggregation, and
the reference arm's rank-0-only rule, in two CPU processes."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        elapsed = [2.0, 3.0][rank]                      # rank 1 is the slow one
        value, el = bench.replica_throughput(elapsed, 16384, 10, "cpu")
        ref_rank0_only = bench.reference_runs_on(rank)
        dist.barrier()
        q.put((rank, value, el, ref_rank0_only))
    finally:
        dist.destroy_process_group()


def test_replica_throughput_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, value, el, ref in got:
        assert el == 3.0                                # the slowest rank's time
        assert value == pytest.approx(2 * 16384 * 10 / 3.0)
        assert ref == (rank == 0)


def test_replica_throughput_single_process():
    sys.path.insert(0, ROOT)
    import bench
    value, el = bench.replica_throughput(2.0, 100, 4, "cpu")
    assert (value, el) == (200.0, 2.0)
