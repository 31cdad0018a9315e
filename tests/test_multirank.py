"""The multi-rank host logic of the benchmark on CPU: two gloo ranks (no GPU).

bench.py runs one process per GPU, each on its own replica of the workload (no collective
on the data path); the only cross-rank steps are the barriers around the timed region and
the max-over-ranks reduction of the step time, which these tests exercise."""
import os
import subprocess
import sys
import tempfile

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, store_file, out):
    # rendezvous through a file store: no TCP port to race for with other processes
    os.environ.update(MASTER_ADDR="127.0.0.1", RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"file://{store_file}", rank=rank, world_size=world)
    try:
        r, w, l = bench.dist_env()
        bench.rank_barrier(w)
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, w, "cpu")
        out[rank] = (r, w, l, ms, bench.job_rate(1000, w, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    store_file = os.path.join(tempfile.mkdtemp(prefix="pisa_pg_"), "store")
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, store_file, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for rank in range(world):
        r, w, l, ms, rate = res[rank]
        assert (r, w, l) == (rank, world, rank)
        assert ms == 15.0                          # the slower rank's time, on every rank
        assert rate == pytest.approx(1000 * world / 0.015)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_rate(10, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
