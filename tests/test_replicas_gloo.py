"""Host logic of the multi-replica benchmark on CPU: two gloo ranks.

Heads and sequences are independent, so N GPUs run N independent replicas
(weak scaling) with no data-path collective; the only cross-rank steps are
the timing barrier and the max-over-ranks reduction of each replica's time.
These tests run that host logic on two CPU processes.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, loc = bench.dist_info()
        dist.barrier()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)   # each replica times its own steps
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.replica_seed(2, rank))
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"info": [r, w, loc], "slowest": slowest, "seeds": seeds}, f)
    finally:
        dist.destroy_process_group()


def test_two_replicas_share_the_slowest_time_and_distinct_batches(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert x["info"] == [r, world, r]
        assert x["slowest"] == 15.0             # max over ranks, seen by every rank
        assert x["seeds"] == [2, 1002]          # each replica draws its own batch
    assert len(set(res[0]["seeds"])) == world


def test_max_over_ranks_without_a_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


@pytest.mark.parametrize("rank", [1])
def test_reference_arm_other_ranks_exit_without_work(rank):
    # under torchrun only rank 0 runs and prints the reference (oracle) line
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
