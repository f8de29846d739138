"""The bench's multi-rank logic (replicas, no data-path collective) with
world_size-2 gloo ranks on CPU: every rank learns the slowest rank's time and
the whole-job value counts the units of all ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [2.0, 3.5][rank]
        ms_max = bench.max_over_ranks(ms_local, "cpu")
        value = bench.whole_job_tflops(1e12, world, ms_max)
        out.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value in res:
        assert ms_max == pytest.approx(3.5)
        assert value == pytest.approx(2 * 1e12 / 3.5e-3 / 1e12)


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.whole_job_tflops(2e12, 1, 1000.0) == pytest.approx(2.0)
