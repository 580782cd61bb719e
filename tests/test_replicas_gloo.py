"""The multi-GPU path is replicas only (independent batches per rank, no data
exchange): its host logic -- per-rank batches, max-over-ranks timing and the
whole-job figure -- checked with two gloo ranks on the CPU, and the reference
arm doing no work on ranks other than 0."""
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads as W
    w = W.SMALL
    # every rank draws its own batch
    q, _, _ = W.qkv(w, H=1, seed=bench.replica_seed(w, rank))
    gathered = [torch.empty_like(q) for _ in range(world)]
    dist.all_gather(gathered, q)
    distinct = not torch.equal(gathered[0], gathered[1])
    # the slowest rank's time is the job's time; work adds over ranks
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
    value = bench.whole_job_tflops(2.0e12, world, ms)
    out[rank] = (distinct, ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_replica_logic():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        distinct, ms, value = res[r]
        assert distinct
        assert ms == 15.0                       # max over ranks, on every rank
        assert abs(value - 2 * 2.0e12 / 15e-3 / 1e12) < 1e-9


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.whole_job_tflops(1.0e12, 1, 1000.0) == 1.0


def test_reference_arm_is_silent_off_rank_zero():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
