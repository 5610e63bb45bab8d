"""The benchmark's N > 1 path on the CPU: two gloo ranks run the replica logic
(every rank decodes its own cache, no data-path collective): per-rank seeds,
the max over ranks of the timed region, the whole-job value, rank 0 alone
printing, and the reference arm doing no work on the other ranks."""
from __future__ import annotations

import contextlib
import io
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    res = {"rank": rank}
    try:
        # the timed region of the slowest rank counts
        res["max"] = bench.max_over_ranks(10.0 + rank, world, "cpu")
        res["seed"] = bench.rank_seed("long128k", rank)
        res["env"] = list(bench.dist_env())
        # reference arm: rank 0 alone times the oracle and prints one line
        sys.argv = ["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                    "--warmup", "1", "--gpus", str(world)]
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(bench.parse())
        res["out"] = buf.getvalue()
        dist.barrier()
    finally:
        dist.destroy_process_group()
    q.put(res)


def test_two_gloo_ranks_replica_logic():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r["rank"]: r for r in results}
    assert by_rank[0]["max"] == by_rank[1]["max"] == 11.0
    assert by_rank[0]["seed"] != by_rank[1]["seed"]
    assert by_rank[0]["env"] == [0, 0, 2] and by_rank[1]["env"] == [1, 1, 2]
    assert by_rank[1]["out"] == ""                          # no work, no line on rank 1
    line = json.loads(by_rank[0]["out"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas each ran K steps within 100 ms of the slowest rank's time
    assert bench.whole_job_us_per_step(0.100, 2) == pytest.approx(50.0)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
