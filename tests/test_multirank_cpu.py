"""The N > 1 host path of the benchmark on CPU: two gloo ranks.

Each rank runs its own replica (weak scaling, no data exchanged); the step
time reported is the slowest rank's, and only rank 0 prints.  Also checks
that the reference arm's non-zero ranks exit without work.
"""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
        got = bench.max_over_ranks(mine, world)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"rank": rank, "max": got}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks(tmp_path):
    port = 29500 + (os.getpid() % 2000)
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        with open(tmp_path / f"rank{r}.json") as f:
            assert json.load(f)["max"] == pytest.approx(15.0)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                         text=True, timeout=300)
    assert res.returncode == 0
    assert res.stdout.strip() == ""
