"""The replica path of bench.py for N > 1 ranks: the step time is the maximum over ranks and
the value is all ranks' work over that time. Runs as 2 gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, "cpu")
    val = bench.whole_job_tflops(1e12, world, ms)
    out.put((rank, ms, val))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2] == pytest.approx(2e12 / 15e-3 / 1e12)


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(2e12, 1, 1000.0) == pytest.approx(2.0)
