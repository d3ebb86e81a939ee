"""The multi-GPU path is data-parallel replicas (tokens are independent; no
collective on the data path).  What crosses ranks is only the benchmark's
timing: the slowest rank's step time, and the whole job's tokens over it.
These run here as two gloo ranks on CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (r + 1) ms per step and 10 * (r + 1) ms end to end
    ms, e2e = bench.max_over_ranks([1.0 + rank, 10.0 * (rank + 1)], world)
    out.put((rank, ms, e2e, bench.whole_job_tokens_per_s(32, world, ms)))
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, e2e, value in res:
        assert ms == 2.0 and e2e == 20.0           # every rank sees the maximum
        assert value == pytest.approx(2 * 32 / 2e-3)  # both ranks' tokens / slowest time


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.whole_job_tokens_per_s(32, 1, 0.25) == pytest.approx(128000.0)
