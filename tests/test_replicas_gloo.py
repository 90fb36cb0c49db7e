"""Host logic of the multi-GPU path on CPU: two gloo ranks.

The fold shards without any exchange (replicas), so the only cross-rank step
is the benchmark's timing: a barrier and the maximum of the step time over
ranks.  Runs as two spawned processes on 127.0.0.1 with the gloo backend."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    step_ms = [0.5, 0.8][rank]  # rank 1 is the slow replica
    slowest = bench.max_over_ranks(step_ms, "cpu")
    dist.barrier()
    q.put((rank, slowest, bench.replica_seed_base(rank),
           bench.job_rows_per_s(512, world, slowest)))
    dist.destroy_process_group()


def test_two_rank_replica_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in results] == [0.8, 0.8]  # both ranks see the max
    assert results[0][2] != results[1][2]  # distinct input seeds per replica
    assert results[0][3] == pytest.approx(2 * 512 / 0.8e-3)


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(1.25, "cpu") == 1.25
