"""The N > 1 path of bench.py on CPU (gloo, world size 2, 127.0.0.1).

The decode path shards into independent replicas (no data-path collective):
under torchrun every rank runs its own work, the timed region is bracketed by
a barrier, and the reported time is the maximum over ranks.  These tests run
that host logic with two gloo ranks, and the reference arm under torchrun,
where rank 0 alone prints the JSON line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, _ = bench.dist_init(world)
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    worst = bench.max_over_ranks(1.5 + rank, w)  # rank 1 is the slower one
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, worst))


def test_max_over_ranks_and_barrier_with_two_gloo_ranks():
    if torch.cuda.is_available():
        pytest.skip("the CPU (gloo) variant of the replica path")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_reference_arm_under_torchrun_prints_once():
    if torch.cuda.is_available():
        pytest.skip("the CPU (gloo) variant of the replica path")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny_gqa_ctx260", "--steps", "2", "--warmup", "1", "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "us"
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    # exactly --steps timed oracle calls (the tiny call fits the CPU budget) after --warmup
    assert d["steps"] == 2 and d["warmup"] == 1 and "2 calls in all" in d["cpu_baseline"]["sample"]
