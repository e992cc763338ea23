"""The N>1 benchmark path on CPU with gloo, world size 2: each rank builds
its own seeded replica (no collective on the data path) and the job's time
is the maximum over ranks."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    w = bench.make_replica("tiny_fp32", rank)
    local_ms = 1.0 + rank  # rank 1 is the slow one
    job_ms = bench.max_over_ranks(local_ms, world)
    # Collect each rank's replica fingerprint on rank 0.
    fp = torch.tensor([float(w.context_lens.sum()), float(w.q.double().sum())], dtype=torch.float64)
    gathered = [torch.zeros_like(fp) for _ in range(world)]
    dist.all_gather(gathered, fp)
    out[rank] = (job_ms, [g.tolist() for g in gathered], bench.job_throughput(1000, world, job_ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_and_max_time():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    job0, fps, thr0 = out[0]
    job1, _, thr1 = out[1]
    assert job0 == job1 == 2.0  # both ranks see the slowest rank's time
    assert fps[0] != fps[1]  # replicas are seeded per rank
    assert thr0 == pytest.approx(2 * 1000 / 2e-3 / 1e9)


def test_reference_arm_prints_only_on_rank_zero(tmp_path):
    import subprocess

    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", "tiny_fp32"], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
