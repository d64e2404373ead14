"""Host-side logic of the benchmark's multi-process path, run as two gloo ranks on the CPU: one process per GPU
reports the whole job's throughput over the slowest rank's time; the reference arm runs on rank 0 only.  The
matmul itself shards with no exchange (each rank multiplies its own matrices), so the ranks meet only at the
barriers around the timed region and in the max over ranks."""
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


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, w)
    bench.barrier(w)
    q.put((rank, slowest, bench.job_throughput(1e9, 100, w, slowest)))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    out = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slowest, gbps in out:
        assert slowest == 15.0                      # the max over ranks, seen by every rank
        assert gbps == pytest.approx(1e9 * 2 * 100 / 15e-3 / 1e9)   # all ranks' bytes over the slowest time


def test_job_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(89e6, 1000, 1, 16.0) == pytest.approx(89e6 * 1000 / 16e-3 / 1e9)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_other_ranks_exit_without_work():
    # under torchrun the reference arm (the CPU oracle) runs on rank 0 only; any other rank exits 0 at once
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
