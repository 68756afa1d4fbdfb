"""The multi-GPU path of the benchmark on the CPU: two gloo ranks run the
host logic of `bench.py --gpus 2` (one replica per rank, weak scaling).

The timed region of each rank is replaced by fixed numbers; the test checks
the cross-rank reduction (the slowest rank's time, the sum of the ranks'
bytes), the whole-job throughput built from it, and that under a two-rank
launch the reference arm prints from rank 0 only.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: device time 10 + 3r ms, end-to-end 20 + 5r ms, 100 (r + 1) bytes a step
        got = bench.aggregate_ranks(10.0 + 3 * rank, 20.0 + 5 * rank, 100 * (rank + 1), world,
                                    "cpu")
        # reference arm under a multi-rank launch: only rank 0 does work and prints
        buf = io.StringIO()
        args = type("A", (), {})()
        with redirect_stdout(buf):
            rc = bench.reference_arm(args, rank, world) if rank != 0 else 0
        dist.barrier()
        results[rank] = (got, rc, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_gpu_job():
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        results = dict(results)
    for rank in range(world):
        (dev_ms, e2e_ms, nbytes), rc, out = results[rank]
        assert dev_ms == pytest.approx(13.0)      # the slower rank's device time
        assert e2e_ms == pytest.approx(25.0)      # and end-to-end time
        assert nbytes == pytest.approx(300.0)     # both replicas' bytes
        assert rc == 0
    assert results[1][2] == ""                    # rank 1 of the reference arm is silent


def test_job_throughput_and_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_ranks(4.0, 5.0, 123, 1, "cpu") == (4.0, 5.0, 123.0)
    # 2 ranks x 1e9 bytes per step, 10 steps in 5 ms -> 4000 GB/s for the job
    assert bench.job_gbs(2e9, 10, 5.0) == pytest.approx(4000.0)
