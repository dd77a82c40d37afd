"""The multi-GPU host logic on CPU: the path does not shard, so every rank runs
an independent replica; the benchmark takes the slowest rank's time and the
units all ranks processed.  Checked with two gloo ranks on the CPU."""
import json
import os
import subprocess
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    sys.path.insert(0, str(ROOT))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    seconds = 1.0 + rank  # rank 1 is the slow one
    units = 100.0 * (rank + 1)
    t, u = bench.aggregate(seconds, units, True)
    bench.barrier(True)
    out[rank] = (t, u)
    dist.destroy_process_group()


def test_aggregate_takes_max_time_and_sum_of_units():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 300.0)


def test_single_rank_aggregate_is_identity():
    sys.path.insert(0, str(ROOT))
    import bench

    assert bench.aggregate(1.5, 42.0, False) == (1.5, 42.0)


@pytest.mark.parametrize("rank", ["1"])
def test_reference_arm_only_rank_zero_prints(rank, tmp_path):
    env = dict(os.environ, RANK=rank, WORLD_SIZE="2", LOCAL_RANK=rank)
    res = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "0"], capture_output=True, text=True,
                         env=env, timeout=300)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_reference_arm_line(tmp_path):
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "0"], capture_output=True, text=True,
                         env=env, timeout=300)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
