"""The multi-rank path of bench.py on CPU (gloo, world size 2): every rank runs
its own replica of the workload (no collective on the data path); the ranks
meet at a barrier around the timed region, the time is the maximum over
ranks, and the whole-job value counts the tokens of every rank."""
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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (rank, world, rank)
        bench.barrier(world)
        per_rank_ms = [120.0, 150.0][rank]  # the ranks finish at different times
        ms = bench.max_over_ranks(per_rank_ms, world)
        value = bench.whole_job_tokens_per_s(4096 * 10, ms, world)
        out.put((rank, ms, value))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_count_every_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, value in got:
        assert ms == 150.0  # the slowest rank's time on every rank
        assert value == pytest.approx(2 * 4096 * 10 / 0.150)  # tokens of both ranks / max time


def test_single_rank_helpers_need_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.whole_job_tokens_per_s(64, 1.0, 1) == pytest.approx(64000.0)


def test_reference_arm_under_two_ranks_prints_once():
    """bench.py --impl reference under torchrun: rank 0 alone times the oracle
    and prints one JSON line; the other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny", "--gpus", "2",
           "--steps", "3", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
