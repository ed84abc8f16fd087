"""The bench's multi-rank host logic on CPU, two gloo ranks (no GPU).

The block shards only as independent replicas: each rank processes its own batch
and there is no collective on the data path.  What the ranks share is the
measurement: the job's time is the slowest rank's, its throughput counts every
rank's tokens, and the reference arm (the oracle on the host cores) runs on rank 0
alone while the other ranks exit without work.
"""

import io
import json
import multiprocessing as mp
import os
import socket
import sys
import types
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, task: str, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if task == "max":
            # rank r took 1 + r ms per step: the job's step is the slowest rank's
            ms = bench.max_over_ranks(1.0 + rank, world)
            out.put((rank, ms, bench.job_throughput(256, world, ms / 1e3)))
        else:
            from expert_routed_ffn_gb300 import workloads as wl
            buf = io.StringIO()
            args = types.SimpleNamespace(steps=2, warmup=1, gpus=world)
            with redirect_stdout(buf):
                bench.run_reference(args, wl.TINY)
            dist.barrier()
            out.put((rank, buf.getvalue(), None))
    finally:
        dist.destroy_process_group()


def _run(task: str, world: int = 2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, task, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def test_job_time_is_the_slowest_rank_and_throughput_counts_every_rank():
    res = _run("max")
    for rank, ms, value in res:
        assert ms == 2.0  # max over ranks, on every rank
        assert value == pytest.approx(2 * 256 / 2e-3)


def test_reference_arm_runs_on_rank_0_only():
    res = _run("reference")
    (r0, out0, _), (r1, out1, _) = res
    assert (r0, r1) == (0, 1)
    assert out1.strip() == ""
    lines = [ln for ln in out0.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
