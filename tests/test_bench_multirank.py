"""Host logic of bench.py with several ranks, run as two gloo processes on CPU.

With N GPUs the benchmark runs one replica per rank (the decode shards by
sequence with no exchange step); the job's time is the slowest rank's total
and the job's throughput counts every rank's tokens.  Only the timing
reduction crosses ranks, so it is exercised here without a GPU.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, totals, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_info()
        dist.barrier()
        total = bench.world_max(torch, totals[rank], "cpu")
        value = bench.job_throughput(w, 1000, 10, total)
        queue.put((r, local, w, total, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_total_and_count_every_rank():
    world, totals = 2, [12.5, 20.0]           # ms of timed steps on each rank
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, totals, queue)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(queue.get(timeout=10) for _ in range(world))
    for r, (rank, local, w, total, value) in enumerate(got):
        assert (rank, local, w) == (r, r, world)
        assert total == max(totals)             # every rank sees the slowest rank's time
        assert value == pytest.approx(world * 1000 * 10 / (max(totals) / 1e3))


def test_single_process_needs_no_process_group():
    assert bench.world_max(torch, 3.5, "cpu") == 3.5
    assert bench.job_throughput(1, 262176, 2000, 100.0) == pytest.approx(262176 * 2000 / 0.1)


def _run_reference(env_extra, tmp_path):
    import json
    import subprocess

    env = dict(os.environ, **env_extra)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                          "--warmup", "3", "--cpu-total-s", "2"], capture_output=True, text=True, env=env,
                         timeout=600, cwd=str(tmp_path))
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    assert _run_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, tmp_path) == []
    (line,) = _run_reference({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"}, tmp_path)
    assert line["impl"] == "reference" and line["unit"] == "KV-tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == (os.cpu_count() or 1)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
