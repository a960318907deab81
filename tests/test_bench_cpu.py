"""Host logic of bench.py that needs no GPU: the max-over-ranks reduction of
the multi-rank run (world size 2 over gloo) and the reference arm's rank
handling (rank 0 prints one JSON line, other ranks exit without work)."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(torch, dist, 10.0 + 5.0 * rank, torch.device("cpu"))
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, 29511, out), nprocs=2, join=True, start_method="spawn")
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, None, 3.5, torch.device("cpu")) == 3.5


def run_bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=env, timeout=600)


def test_reference_arm_non_zero_rank_exits_quietly():
    r = run_bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference", "--steps", "1",
                  "--warmup", "3")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = run_bench({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"}, "--impl", "reference", "--steps", "1",
                  "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOPS" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0
