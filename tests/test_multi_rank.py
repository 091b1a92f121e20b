"""The multi-rank path of bench.py on the CPU (gloo, world size 2): the whole-job
timing is the slowest rank's, throughput counts every rank's work, and the
reference arm under torchrun prints exactly one line from rank 0 while the other
rank exits without work.  Token rows shard with no exchange, so replicas are
the only multi-GPU mode; nothing here touches a GPU."""
import json
import os
import socket
import subprocess
import sys
import tempfile

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank "timed" a different step; everyone must report the slowest
        ms = bench.max_over_ranks(dist, 10.0 + 7.0 * rank, "cpu")
        tops = bench.whole_job_tops(world, ms)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "tops": tops}, f)
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_every_rank_counts():
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(world, _free_port(), d), nprocs=world,
                           start_method="spawn")
        got = [json.load(open(os.path.join(d, f"rank{r}.json"))) for r in range(world)]
    assert all(g["ms"] == 17.0 for g in got)
    expect = world * bench.step_ops() / 17e-3 / 1e12
    assert all(abs(g["tops"] - expect) <= 1e-9 * expect for g in got)
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0
