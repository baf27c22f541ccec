"""The benchmark's multi-rank host path on CPU: two gloo ranks (one process each, started
with spawn) run the process-group set-up, the max-over-ranks timing reduction, the
barrier and the reference arm's rank gating (rank 0 alone runs the oracle, here on a small
decode of 2 requests x 2,048 entries, and prints the line).  Decode requests are independent, so the replicas exchange nothing
else; the seeds of their requests must not overlap."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch
    import bench
    res = {}
    try:
        ws, r, local = bench.dist_init()
        res["ws"], res["rank"] = ws, r
        res["max"] = bench.max_over_ranks(10.0 * r + 0.25, ws)  # slowest rank's time wins
        bench.barrier(ws)
        sys.argv = ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
                    "--batch", "2", "--ctx", "2048"]
        args = bench.parse()
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(args, ws, r, local)
        res["out"] = buf.getvalue()
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    except Exception as exc:  # reported to the parent
        res["error"] = f"{type(exc).__name__}: {exc}"
    q.put(res)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="the CPU gloo path; GPU runs use NCCL")
def test_two_gloo_ranks_reduce_and_gate_output():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res = sorted(res, key=lambda d: d.get("rank", -1))
    assert all("error" not in d for d in res), res
    assert [d["ws"] for d in res] == [2, 2] and [d["rank"] for d in res] == [0, 1]
    assert [d["max"] for d in res] == [10.25, 10.25]
    assert res[1]["out"] == ""                              # only rank 0 prints
    line = json.loads(res[0]["out"].strip())
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_replica_seeds_do_not_overlap():
    sys.path.insert(0, ROOT)
    import bench
    B = 128
    seeds = []
    for rank in range(8):
        base = bench.rank_seed_base(rank)
        seeds.append(set(range(base, base + B)) | set(range(base + 50000, base + 50000 + B)) |
                     set(range(base + 7_000_000, base + 7_000_000 + 8)))
    for i in range(8):
        for j in range(i + 1, 8):
            assert not seeds[i] & seeds[j]
