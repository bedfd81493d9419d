"""The benchmark's multi-rank plumbing on CPU: two gloo ranks.

The path runs as independent replicas (one per GPU, no collective on the
data path); what N > 1 adds is host logic: process-group set-up from the
launcher's environment, the barrier around the timed region, the maximum
of the per-rank times, and only rank 0 running the reference arm.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "CUDA_VISIBLE_DEVICES": ""})
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + rank, w)
    # the reference arm: every rank but 0 returns at once, without work
    ran = None
    if rank != 0:
        class A:
            steps, warmup, gpus, ref_step_seconds = 1, 0, world, 0.5
        bench.run_reference(A, rank, w)
        ran = "returned"
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((rank, slowest, ran))


@pytest.mark.timeout(120)
def test_two_gloo_ranks_share_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.5, None), (1, 2.5, "returned")]
