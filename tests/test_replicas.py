"""Multi-process host logic of the benchmark (CPU, gloo, world size 2).

The path shards into independent replicas: each rank streams its own copy of
the workload and nothing crosses ranks but the timing reduction.  These tests
run that reduction on two gloo ranks: the job time is the slowest rank's, the
job's bytes are the sum over ranks, and the reference arm does no work on any
rank but 0.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r ran (r+1) ms and streamed (r+1) GB
        ms, gbs = bench.replica_aggregate(1.0 + rank, 1e9 * (1 + rank), dist, "cpu")
        out.put((rank, ms, gbs))
    finally:
        dist.destroy_process_group()


def test_replica_aggregate_two_ranks():
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
    # max time = 2 ms, total bytes = 3 GB -> 1500 GB/s, the same on both ranks
    for rank, ms, gbs in res:
        assert ms == pytest.approx(2.0)
        assert gbs == pytest.approx(3e9 / 2e-3 / 1e9)


def test_replica_aggregate_single_process():
    sys.path.insert(0, ROOT)
    import bench

    ms, gbs = bench.replica_aggregate(4.0, 2e9)
    assert ms == 4.0 and gbs == pytest.approx(500.0)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_json_line():
    """The reference arm (the scalar CPU oracle on a bounded sample) prints one
    JSON line with the contract's keys, on the host cores only."""
    import json

    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]

