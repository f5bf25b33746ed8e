"""The benchmark's multi-process path on CPU (gloo, world size 2): the
element-wise maximum of the ranks' times, the whole-job rate built from it,
and the reference arm launched as two ranks by torch.distributed.run (rank 0
alone measures and prints one line; the other exits cleanly). The GPU arm
uses the same functions over NCCL."""
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
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r took (1 + r) s for the step, (3 - r) s end to end.
        got = bench.max_over_ranks([1.0 + rank, 3.0 - rank, 0.5], dist)
        out.put((rank, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world_2_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    results = dict(out.get() for _ in range(2))
    assert results[0] == results[1] == [2.0, 3.0, 0.5]


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], None) == [1.5, 2.5]


def test_whole_job_rate_is_weak_scaling_over_the_slowest_rank():
    # 2 GB a step, 10 steps in 1 s on the slowest of 4 ranks: 80 GB/s in all.
    assert bench.whole_job_rate(2e9, 10, 4, 1.0) == pytest.approx(80.0)
    assert bench.whole_job_rate(2e9, 10, 1, 1.0) == pytest.approx(20.0)


def test_reference_arm_as_two_ranks():
    """`python -m torch.distributed.run --nproc-per-node 2 bench.py --impl
    reference`: one JSON line (rank 0), both ranks exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--ref-budget", "0.3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
