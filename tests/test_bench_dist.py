"""The multi-rank host logic of bench.py on CPU with gloo (world size 2).

The path does not shard across GPUs (replicas only): each rank times its own
replica and rank 0 reports the slowest rank's time.  Here two CPU ranks check
that reduction; the reference arm's non-zero ranks do no work.
"""

import os
import subprocess
import sys
import tempfile

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, store_file, results):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    # a file rendezvous: no TCP port to race for
    dist.init_process_group("gloo", init_method=f"file://{store_file}", rank=rank, world_size=world)
    local = [3.5, 7.25][rank]
    results[rank] = bench.max_over_ranks(local, dist)
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_time_is_reported():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    store_file = os.path.join(tempfile.mkdtemp(), "rendezvous")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, store_file, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {0: 7.25, 1: 7.25}


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5) == 2.5


def test_reference_arm_nonzero_rank_does_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
