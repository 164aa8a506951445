"""The bench's multi-GPU path is replicas (one drafter per GPU, no data-path
collective): its host logic -- rank discovery, max-over-ranks timing, the
whole-job throughput, rank 0 alone running the reference arm -- checked
with two gloo ranks on CPU."""
import os
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, local, w = bench.dist_env()
        ms = bench.max_over_ranks(10.0 + 2.5 * rank, w, "cpu")   # rank 1 is the slow one
        value = bench.job_throughput(w, 16, 200, ms)

        class Args:
            workload = "tiny_f32_L1_N128"
            warmup, steps = 1, 1
        ran = bench.run_reference(Args()) if rank != 0 else None   # non-zero ranks exit at once
        q.put((r, local, w, ms, value, ran))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_whole_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    env_pp = os.environ.get("PYTHONPATH", "")
    os.environ["PYTHONPATH"] = ROOT + (os.pathsep + env_pp if env_pp else "")
    try:
        for p in procs:
            p.start()
        got = sorted(q.get(timeout=120) for _ in procs)
        for p in procs:
            p.join(timeout=60)
            assert p.exitcode == 0
    finally:
        os.environ["PYTHONPATH"] = env_pp
        for p in procs:
            if p.is_alive():
                p.kill()
    for r, (rank, local, world, ms, value, ran) in enumerate(got):
        assert (rank, local, world) == (r, r, 2)
        assert ms == pytest.approx(12.5)                       # the slowest rank's time, on both
        assert value == pytest.approx(2 * 16 * 200 / 12.5e-3)  # both replicas' drafted tokens
        assert ran is None
