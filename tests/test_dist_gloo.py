"""Multi-process host logic of the benchmark with the gloo backend (CPU).

The decode path has no exchange step: N > 1 runs N independent replicas,
and only the timing reduction (max over ranks), the byte count (sum over
ranks) and the barriers cross processes.  These run here on CPU ranks.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.init_dist("gloo")
    try:
        assert bench._dist_on()
        bench.barrier()
        mx = bench.reduce_over_ranks(10.0 + rank, "max")
        sm = bench.reduce_over_ranks(1.0 + rank, "sum")
        gbs, ms = bench.aggregate(1e9 * (rank + 1), 100.0 * (rank + 1))
        q.put((rank, mx, sm, gbs, ms))
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()


def test_reductions_and_aggregate_world2():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, mx, sm, gbs, ms in res:
        assert mx == 11.0 and sm == 3.0
        # (1e9 + 2e9) bytes over the slowest rank's 200 ms = 15 GB/s
        assert ms == 200.0 and abs(gbs - 15.0) < 1e-9


def test_single_process_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.5, "max") == 3.5
    gbs, ms = bench.aggregate(2e9, 1000.0)
    assert gbs == 2.0 and ms == 1000.0


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--workload", "fp16_4096"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0 and p.stdout.strip() == ""


def test_reference_arm_prints_one_line():
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--workload", "fp16_4096"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
