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


def _ring_worker(rank, world, port, causal, q):
    """Ring attention over 2 ranks with the oracle standing in for the kernels (fp64, CPU): checks
    the ring's schedule, rotation and merge against whole-sequence attention."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np

        import oracle
        from exact_io_aware_38_gb300 import ring

        g = torch.Generator().manual_seed(5)
        B, N, H, d = 1, 2 * 48, 2, 8
        full = [torch.randn((B, N, H, d), generator=g, dtype=torch.float64) for _ in range(3)]
        blk = N // world
        qb, kb, vb = (t[:, rank * blk:(rank + 1) * blk].contiguous() for t in full)
        t4 = lambda x: x.numpy().transpose(0, 2, 1, 3)

        def partial(q_, k_, v_, c_):
            o, lse = oracle.attention_forward(t4(q_), t4(k_), t4(v_), 0.35, causal=c_)
            return torch.from_numpy(o), torch.from_numpy(lse)

        def merge(acc, part):
            (oa, la), (op, lp) = acc, part
            m = torch.maximum(la, lp)
            wa = torch.where(torch.isinf(la), torch.zeros_like(la), torch.exp(la - m))
            wp = torch.where(torch.isinf(lp), torch.zeros_like(lp), torch.exp(lp - m))
            o = (wa[..., None] * oa + wp[..., None] * op) / (wa + wp)[..., None]
            return o, m + torch.log(wa + wp)

        o, lse = ring.ring_forward(qb, kb, vb, causal=causal, partial=partial, merge=merge, finalize=lambda a: a)
        ref_o, ref_l = oracle.attention_forward(t4(full[0]), t4(full[1]), t4(full[2]), 0.35, causal=causal)
        err_o = float(np.abs(o.numpy() - ref_o[:, :, rank * blk:(rank + 1) * blk]).max())
        err_l = float(np.abs(lse.numpy() - ref_l[:, :, rank * blk:(rank + 1) * blk]).max())
        q.put((rank, err_o, err_l))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_two_ranks(causal):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ring_worker, args=(r, 2, port, causal, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err_o, err_l in results:
        assert err_o <= 1e-12 and err_l <= 1e-12, (rank, err_o, err_l)


def _ring_bwd_worker(rank, world, port, causal, q):
    """Ring backward over `world` ranks with the oracle's per-block share standing in for the
    kernel (fp64, CPU): checks the rotation of the dK/dV accumulators and the final delivery
    against whole-sequence gradients."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np

        import oracle
        from exact_io_aware_38_gb300 import ring

        g = torch.Generator().manual_seed(7)
        B, N, H, Hkv, d, c = 1, world * 20, 4, 2, 6, 0.35
        qf = torch.randn((B, N, H, d), generator=g, dtype=torch.float64)
        kf, vf = (torch.randn((B, N, Hkv, d), generator=g, dtype=torch.float64) for _ in range(2))
        dof = torch.randn((B, N, H, d), generator=g, dtype=torch.float64)
        t4 = lambda x: np.ascontiguousarray(x.numpy().transpose(0, 2, 1, 3))
        back = lambda a: torch.from_numpy(np.ascontiguousarray(a.transpose(0, 2, 1, 3)))
        of, lf = oracle.attention_forward(t4(qf), t4(kf), t4(vf), c, causal=causal)
        blk = N // world
        sl = slice(rank * blk, (rank + 1) * blk)
        qb, kb, vb, dob = (t[:, sl].contiguous() for t in (qf, kf, vf, dof))
        ob, lb = back(of)[:, sl].contiguous(), torch.from_numpy(lf[:, :, sl].copy())

        def partial_bwd(q_, k_, v_, o_, l_, do_, c_, aq, ak, av):
            gq, gk, gv = oracle.attention_backward_block(t4(q_), t4(k_), t4(v_), t4(o_), l_.numpy(), t4(do_), c,
                                                         causal=c_)
            aq += back(gq)
            ak += back(gk)
            av += back(gv)

        dq, dk, dv = ring.ring_backward(qb, kb, vb, ob, lb, dob, causal=causal, partial_bwd=partial_bwd)
        rq, rk, rv = (back(x)[:, sl] for x in oracle.attention_backward(t4(qf), t4(kf), t4(vf), t4(dof), c,
                                                                         causal=causal))
        q.put((rank, float((dq - rq).abs().max()), float((dk - rk).abs().max()), float((dv - rv).abs().max())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_backward(causal, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ring_bwd_worker, args=(r, world, port, causal, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, eq, ek, ev in results:
        assert max(eq, ek, ev) <= 1e-12, (rank, eq, ek, ev)


def test_ring_schedule_covers_each_block_once():
    from exact_io_aware_38_gb300 import ring

    for world in (1, 2, 3, 5):
        for rank in range(world):
            for causal in (False, True):
                sched = ring.ring_schedule(rank, world, causal)
                assert sorted(src for _, src, _ in sched) == list(range(world))
                used = {src: c for _, src, c in sched}
                assert used[rank] is causal  # own block: causal (square) or whole
                for src, c in used.items():
                    if src < rank:
                        assert c is False
                    elif src > rank:
                        assert c is (None if causal else False)
