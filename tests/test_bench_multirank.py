"""The N>1 bench path on CPU: two gloo ranks, each timing its own replica;
the reported time is the slowest rank's, and no data-path collective runs."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + rank, w)      # rank 1 is the slow one
    q.put((rank, slowest))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert not dist.is_initialized()


def test_step_flops_closed_form():
    """4Mkn + 2Mr(k+n) + 2Mr(2n+3k) for one 512x512 projection at M=256, r=8."""
    import bench
    from lora_inputs import WORKLOADS
    M, k, n, r = 256, 512, 512, 8
    want = 4 * M * k * n + 2 * M * r * (k + n) + 2 * M * r * (2 * n + 3 * k)
    assert bench.step_flops(WORKLOADS["single_512"], M) == want
