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


_RANK_SCRIPT = """
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank, local_rank, world = bench.env_rank()
dist.init_process_group("gloo")
ms = bench.max_over_ranks([1.0 + rank], world)[0]
if rank == 0:
    print(json.dumps({{"world": world, "ms": ms,
                      "value": bench.whole_job_tokens_per_s(32, world, ms)}}), flush=True)
dist.destroy_process_group()
"""


def test_launcher_starts_ranks_under_torchrun(tmp_path):
    """bench.py --gpus N without torchrun's environment re-runs itself under
    torch.distributed.run with N ranks on 127.0.0.1; the same command, pointed
    at a small rank script, brings up two gloo ranks that see WORLD_SIZE = 2."""
    import json
    import subprocess
    import sys

    import bench
    port = _free_port()
    cmd = bench.launcher_command(["--gpus", "2", "--steps", "3"], 2, port)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=2" in cmd and ["--master-addr", "127.0.0.1"] == cmd[5:7]
    assert cmd[-4:] == ["--gpus", "2", "--steps", "3"]
    assert cmd[-5].endswith("bench.py")
    script = tmp_path / "rank.py"
    script.write_text(_RANK_SCRIPT.format(root=os.path.dirname(os.path.abspath(bench.__file__))))
    cmd = cmd[:-5] + [str(script)]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    env.pop("WORLD_SIZE", None)
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=180, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads([ln for ln in res.stdout.splitlines() if ln.startswith("{")][-1])
    assert line["world"] == 2 and line["ms"] == 2.0
    assert line["value"] == pytest.approx(2 * 32 / 2e-3)
