"""The multi-GPU path of the benchmark is N independent replicas: no data
moves between ranks, and the only collective is the MAX of the step times
(the slowest replica bounds the job).  These tests run it on the CPU as two
gloo processes, and check that the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, step_ms, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(step_ms[rank], world, torch.device("cpu"))
        out.put((rank, m, bench.aggregate_value(1.0e9, world, m)))
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_slowest_replica():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    step_ms = [2.0, 5.0]
    procs = [ctx.Process(target=_replica, args=(r, 2, port, step_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, m, v in res:
        assert m == 5.0, "every rank sees the slowest replica's time"
        assert v == pytest.approx(2 * 1.0e9 / 5.0e-3 / 1e9), "value = both replicas' bytes / slowest time"


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.aggregate_value(2.0e9, 1, 4.0) == pytest.approx(500.0)


def _reference(rank: int):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                           "--steps", "2", "--warmup", "3", "--workload", "tiny"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_other_ranks_exit_without_work():
    r = _reference(1)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = _reference(0)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["name"] == "tiny"
