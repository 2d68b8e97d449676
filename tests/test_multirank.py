"""The multi-GPU path of the benchmark, on CPU with gloo (world size 2).

Attention over independent (batch, head) problems shards with no data-path collective: each rank
runs its own batch (weak scaling) and the only exchange is the max-over-ranks reduction of the
step time. This checks that reduction and that the ranks draw different seeded batches."""

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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from exact_io_aware_38_gb300 import workloads

        got = bench.max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
        w = workloads.WORKLOADS["c4"]
        inp = workloads.make_inputs(w, H=1, N=256, seed=w.seed + rank)
        s = torch.tensor([float(inp["q"].float().sum())])
        gathered = [torch.zeros(1) for _ in range(world)]
        dist.all_gather(gathered, s)
        q.put((rank, got, [float(g) for g in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    for rank, got, sums in results:
        assert got == pytest.approx(2.5)  # max over ranks of 1.5 + rank
        assert sums[0] != sums[1]         # replicas run different seeded batches
    assert results[0][2] == results[1][2]


def test_single_process_max_is_identity():
    import bench

    assert bench.max_over_ranks(3.25, None, torch.device("cpu")) == 3.25
