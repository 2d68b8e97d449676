"""GPU parity for strided, unequal-length and packed batches (fa_fwd_varlen / fa_bwd_varlen)
against the fp64 oracle, with the tolerances of test_gpu_parity.py. Causal attention is aligned to
the bottom-right corner (key j visible to query i iff j <= i + L_k - L_q)."""

import numpy as np
import pytest
import torch

import exact_io_aware_38_gb300 as fa
import oracle
from exact_io_aware_38_gb300 import build, workloads

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX, REL_FRO = 2e-2, 2e-3, 1e-3, 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    fa.lib()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def f64(t):
    return t.detach().double().cpu().numpy()


def bf16(shape, g, std=1.0):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def check_o_lse(o, lse, o_ref, lse_ref):
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    empty = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == empty).all()
    if (~empty).any():
        assert np.abs(lse[~empty] - lse_ref[~empty]).max() <= LSE_MAX


def rel_fro(x, ref):
    nr = np.linalg.norm(ref)
    if nr == 0:
        assert np.abs(x).max() <= 1e-3
        return 0.0
    r = np.linalg.norm(x - ref) / nr
    assert r <= REL_FRO, r
    return r


def run_status(fn):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fn(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_bshd_views_match_contiguous_path(causal, d):
    """The same problem through fa_fwd/fa_bwd ([B, H, N, d]) and through the strided entry on a
    [B, N, H, d] copy: identical O, LSE, dK, dV bits (same tiles, same order); dQ to rounding."""
    g = torch.Generator().manual_seed(31 + d)
    B, H, N = 2, 4, 300
    q, k, v, do = (bf16((B, H, N, d), g).cuda() for _ in range(4))
    o1, l1 = fa.fwd(q, k, v, causal=causal)
    dq1, dk1, dv1 = fa.bwd(q, k, v, o1, l1, do, causal=causal)
    qs, ks, vs, dos = (t.transpose(1, 2).contiguous() for t in (q, k, v, do))  # [B, N, H, d]
    o2, l2 = run_status(lambda st: fa.fwd_varlen(qs, ks, vs, causal=causal, status=st))
    dq2, dk2, dv2 = run_status(lambda st: fa.bwd_varlen(qs, ks, vs, o2, l2, dos, causal=causal, status=st))
    assert torch.equal(o1, o2.transpose(1, 2)) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2.transpose(1, 2)) and torch.equal(dv1, dv2.transpose(1, 2))
    assert (dq1.float() - dq2.transpose(1, 2).float()).abs().max() <= 1e-2


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 100), (1, 257), (257, 1), (129, 129), (64, 640)])
def test_unequal_lengths(Nq, Nk, d, causal):
    g = torch.Generator().manual_seed(Nq * 7 + Nk + d)
    B, H, Hkv = 2, 4, 2
    q, do = bf16((B, Nq, H, d), g), bf16((B, Nq, H, d), g)
    k, v = bf16((B, Nk, Hkv, d), g), bf16((B, Nk, Hkv, d), g)
    scale = 1.0 / np.sqrt(d)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = run_status(lambda st: fa.fwd_varlen(qc, kc, vc, causal=causal, scale=scale, status=st))
    dq, dk, dv = run_status(lambda st: fa.bwd_varlen(qc, kc, vc, o, lse, doc, causal=causal, scale=scale, status=st))
    t4 = lambda x: f64(x).transpose(0, 2, 1, 3)  # [B, N, H, d] -> [B, H, N, d]
    ro, rl = oracle.attention_forward(t4(q), t4(k), t4(v), scale, causal=causal)
    check_o_lse(t4(o), f64(lse), ro, rl)
    rdq, rdk, rdv = oracle.attention_backward(t4(q), t4(k), t4(v), t4(do), scale, causal=causal)
    rel_fro(t4(dq), rdq)
    rel_fro(t4(dk), rdk)
    rel_fro(t4(dv), rdv)


PACKED = [
    ([5, 0, 131, 300, 1], [9, 4, 131, 257, 128]),
    ([128, 256, 77], [128, 256, 77]),
    ([640], [1000]),
    ([3, 200, 129, 1, 0, 64], [300, 2, 129, 1, 5, 70]),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", range(len(PACKED)))
def test_packed_sequences(case, d, causal):
    lq, lk = PACKED[case]
    g = torch.Generator().manual_seed(100 + case * 3 + d)
    H, Hkv = 4, 2
    cu_q = np.cumsum([0] + lq).astype(np.int32)
    cu_k = np.cumsum([0] + lk).astype(np.int32)
    rows_q, rows_k = int(cu_q[-1]) + 5, int(cu_k[-1]) + 3  # spare rows outside every sequence
    q, do = bf16((rows_q, H, d), g), bf16((rows_q, H, d), g)
    k, v = bf16((rows_k, Hkv, d), g), bf16((rows_k, Hkv, d), g)
    scale = 1.0 / np.sqrt(d)
    cq, ck = torch.tensor(cu_q, device="cuda"), torch.tensor(cu_k, device="cuda")
    mq, mk = max(max(lq), 1) + 37, max(max(lk), 1)  # the bound may exceed every length
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    sentinel = torch.full_like(qc, float("nan"))
    lse0 = torch.full((H, rows_q), 7.0, device="cuda")
    dk0, dv0 = torch.full_like(kc, 3.0), torch.full_like(vc, 3.0)
    o, lse = run_status(lambda st: fa.fwd_varlen(qc, kc, vc, cq, ck, mq, mk, causal=causal, scale=scale,
                                                 out=sentinel, lse=lse0, status=st))
    dq, dk, dv = run_status(lambda st: fa.bwd_varlen(qc, kc, vc, o, lse, doc, cq, ck, mq, mk, causal=causal,
                                                     scale=scale, dk=dk0, dv=dv0, status=st))
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    # rows outside every sequence are never written (dQ's are set to zero)
    assert torch.isnan(o[tq:].float()).all() and (lse[:, tq:] == 7.0).all()
    assert (dk[tk:].float() == 3.0).all() and (dv[tk:].float() == 3.0).all()
    assert (dq[tq:].float() == 0).all()
    ro, rl = oracle.attention_forward_varlen(f64(q), f64(k), f64(v), cu_q, cu_k, scale, causal=causal)
    check_o_lse(f64(o)[:tq], f64(lse)[:, :tq], ro[:tq], rl[:, :tq])
    rdq, rdk, rdv = oracle.attention_backward_varlen(f64(q), f64(k), f64(v), f64(do), cu_q, cu_k, scale,
                                                     causal=causal)
    rel_fro(f64(dq)[:tq], rdq[:tq])
    rel_fro(f64(dk)[:tk], rdk[:tk])
    rel_fro(f64(dv)[:tk], rdv[:tk])


def test_packed_long_causal_sampled():
    """A packed batch at length 8192 (the long-context shape, 4 heads, two sequences of unequal
    query/key lengths), checked on sampled rows and key columns per sequence."""
    g = torch.Generator().manual_seed(9)
    H, d = 4, 128
    lq, lk = [8192, 3000], [8192, 5000]
    cu_q, cu_k = np.cumsum([0] + lq).astype(np.int32), np.cumsum([0] + lk).astype(np.int32)
    q, do = bf16((cu_q[-1], H, d), g), bf16((cu_q[-1], H, d), g)
    k, v = bf16((cu_k[-1], H, d), g), bf16((cu_k[-1], H, d), g)
    scale = 1.0 / np.sqrt(d)
    cq, ck = torch.tensor(cu_q, device="cuda"), torch.tensor(cu_k, device="cuda")
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = run_status(lambda st: fa.fwd_varlen(qc, kc, vc, cq, ck, 8192, 8192, causal=True, scale=scale, status=st))
    dq, dk, dv = run_status(lambda st: fa.bwd_varlen(qc, kc, vc, o, lse, doc, cq, ck, 8192, 8192, causal=True,
                                                     scale=scale, status=st))
    rng = np.random.default_rng(3)
    for b in range(2):
        sq, sk = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        h = b * 3
        qh, kh, vh, doh = f64(q[sq, h]), f64(k[sk, h]), f64(v[sk, h]), f64(do[sq, h])
        rows = np.sort(rng.choice(lq[b], 200, replace=False))
        cols = np.sort(rng.choice(lk[b], 200, replace=False))
        om, lm = oracle.head_forward(qh, kh, vh, scale, True, rows=rows)
        check_o_lse(f64(o[sq, h])[rows], f64(lse[h, sq])[rows], om, lm)
        rel_fro(f64(dq[sq, h])[rows], oracle.head_dq(qh, kh, vh, doh, scale, True, rows=rows))
        rdk, rdv = oracle.head_dkdv(qh, kh, vh, doh, scale, True, cols=cols)
        rel_fro(f64(dk[sk, h])[cols], rdk)
        rel_fro(f64(dv[sk, h])[cols], rdv)


@pytest.mark.parametrize("d", [64, 128])
def test_splitkv_one_split_equals_unsplit(d):
    """One split runs the partial pass and the merge; its O and LSE equal the plain forward bits."""
    g = torch.Generator().manual_seed(50 + d)
    q, k, v = bf16((2, 130, 4, d), g).cuda(), bf16((2, 700, 2, d), g).cuda(), bf16((2, 700, 2, d), g).cuda()
    o1, l1 = fa.fwd_varlen(q, k, v, causal=True)
    o2, l2 = run_status(lambda st: fa.fwd_splitkv(q, k, v, num_splits=1, causal=True, status=st))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk,splits", [(1, 2049, 5), (7, 300, 2), (1, 1, 3), (128, 1000, 64), (200, 8192, 16),
                                          (1, 8192, None)])
def test_splitkv_decode_shapes(Nq, Nk, splits, d, causal):
    g = torch.Generator().manual_seed(Nq + Nk + d)
    B, H, Hkv = 2, 8, 2
    q = bf16((B, Nq, H, d), g)
    k, v = bf16((B, Nk, Hkv, d), g), bf16((B, Nk, Hkv, d), g)
    scale = 1.0 / np.sqrt(d)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = run_status(lambda st: fa.fwd_splitkv(qc, kc, vc, num_splits=splits, causal=causal, scale=scale,
                                                  status=st))
    t4 = lambda x: f64(x).transpose(0, 2, 1, 3)
    ro, rl = oracle.attention_forward(t4(q), t4(k), t4(v), scale, causal=causal)
    check_o_lse(t4(o), f64(lse), ro, rl)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(12, 3), (32, 1)])
def test_decode_grouped_heads_equal_repeated_kv(H, Hkv, d, causal):
    """One query row per head with grouped K/V heads runs as G rows of each K/V head (one query
    tile per K/V head). Its O and LSE must equal, bit for bit, the same problem with the K/V heads
    repeated, which runs one query row per head; and match the oracle."""
    g = torch.Generator().manual_seed(H * 7 + d)
    B, Nk = 3, 1000
    q = bf16((B, 1, H, d), g)
    k, v = bf16((B, Nk, Hkv, d), g), bf16((B, Nk, Hkv, d), g)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = run_status(lambda st: fa.fwd_varlen(qc, kc, vc, causal=causal, status=st))
    kr, vr = (x.repeat_interleave(H // Hkv, dim=2).contiguous() for x in (kc, vc))
    o2, l2 = run_status(lambda st: fa.fwd_varlen(qc, kr, vr, causal=causal, status=st))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    t4 = lambda x: f64(x).transpose(0, 2, 1, 3)
    ro, rl = oracle.attention_forward(t4(q), t4(k), t4(v), 1.0 / np.sqrt(d), causal=causal)
    check_o_lse(t4(o1), f64(l1), ro, rl)


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_packed(causal):
    lq, lk = [1, 4, 0, 1, 130], [5000, 900, 7, 1, 2000]
    g = torch.Generator().manual_seed(77)
    H, Hkv, d = 8, 4, 128
    cu_q, cu_k = np.cumsum([0] + lq).astype(np.int32), np.cumsum([0] + lk).astype(np.int32)
    q = bf16((cu_q[-1] + 2, H, d), g)
    k, v = bf16((cu_k[-1], Hkv, d), g), bf16((cu_k[-1], Hkv, d), g)
    cq, ck = torch.tensor(cu_q, device="cuda"), torch.tensor(cu_k, device="cuda")
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / np.sqrt(d)
    out = torch.full_like(qc, float("nan"))
    o, lse = run_status(lambda st: fa.fwd_splitkv(qc, kc, vc, cq, ck, max(lq), max(lk), num_splits=9, causal=causal,
                                                  scale=scale, out=out, status=st))
    tq = int(cu_q[-1])
    assert torch.isnan(o[tq:].float()).all()
    ro, rl = oracle.attention_forward_varlen(f64(q), f64(k), f64(v), cu_q, cu_k, scale, causal=causal)
    check_o_lse(f64(o)[:tq], f64(lse)[:, :tq], ro[:tq], rl[:, :tq])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_ring_attention_simulated_on_one_gpu(causal, d):
    """The ring's per-rank schedule run on one GPU with the library's partial, merge and finalize
    kernels (4 blocks of 300 rows, K/V heads shared by two query heads), against the oracle."""
    from exact_io_aware_38_gb300 import ring

    g = torch.Generator().manual_seed(200 + d)
    W, blk, B, H, Hkv = 4, 300, 1, 4, 2
    q = bf16((B, W * blk, H, d), g)
    k, v = bf16((B, W * blk, Hkv, d), g), bf16((B, W * blk, Hkv, d), g)
    scale = 1.0 / np.sqrt(d)
    t4 = lambda x: f64(x).transpose(0, 2, 1, 3)
    ro, rl = oracle.attention_forward(t4(q), t4(k), t4(v), scale, causal=causal)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    block = lambda t, i: t[:, i * blk:(i + 1) * blk].contiguous()
    for rank in range(W):
        qb = block(qc, rank)
        acc = None
        for _, src, c in ring.ring_schedule(rank, W, causal):
            if c is None:
                continue
            part = fa.fwd_partial(qb, block(kc, src), block(vc, src), causal=c, scale=scale)
            acc = part if acc is None else fa.merge_partials(qb, block(kc, src), acc, part)
        o, lse = fa.finalize_partials(qb, block(kc, rank), acc)
        torch.cuda.synchronize()
        sl = slice(rank * blk, (rank + 1) * blk)
        check_o_lse(t4(o), f64(lse), ro[:, :, sl], rl[:, :, sl])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_ring_backward_simulated_on_one_gpu(causal, d):
    """The ring backward's per-rank schedule on one GPU: each (query block, key block) share from
    the library's backward with the rows' final O and LSE (from the ring forward), dQ summed per
    query block and dK, dV per key block in fp32, against the whole-sequence oracle gradients."""
    from exact_io_aware_38_gb300 import ring

    g = torch.Generator().manual_seed(300 + d)
    W, blk, B, H, Hkv = 3, 260, 1, 4, 2
    q, do = bf16((B, W * blk, H, d), g), bf16((B, W * blk, H, d), g)
    k, v = bf16((B, W * blk, Hkv, d), g), bf16((B, W * blk, Hkv, d), g)
    scale = 1.0 / np.sqrt(d)
    t4 = lambda x: f64(x).transpose(0, 2, 1, 3)
    rq, rk, rv = oracle.attention_backward(t4(q), t4(k), t4(v), t4(do), scale, causal=causal)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    block = lambda t, i: t[:, i * blk:(i + 1) * blk].contiguous()
    dq = torch.zeros((B, W * blk, H, d), dtype=torch.float32, device="cuda")
    dk = torch.zeros((B, W * blk, Hkv, d), dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    dq16, dk16, dv16 = torch.zeros_like(dq), torch.zeros_like(dk), torch.zeros_like(dv)  # bf16 shares summed
    for rank in range(W):
        qb, dob = block(qc, rank), block(doc, rank)
        acc = None
        for _, src, c in ring.ring_schedule(rank, W, causal):
            if c is None:
                continue
            part = fa.fwd_partial(qb, block(kc, src), block(vc, src), causal=c, scale=scale)
            acc = part if acc is None else fa.merge_partials(qb, block(kc, src), acc, part)
        ob, lb = fa.finalize_partials(qb, block(kc, rank), acc)
        for _, src, c in ring.ring_schedule(rank, W, causal):
            if c is None:
                continue
            # fp32 shares added in place into the accumulators' blocks (views of the full tensors)
            fa.bwd_varlen_accumulate(qb, block(kc, src), block(vc, src), ob, lb, dob, dq[:, rank * blk:(rank + 1) * blk],
                                     dk[:, src * blk:(src + 1) * blk], dv[:, src * blk:(src + 1) * blk], causal=c,
                                     scale=scale)
            gq, gk, gv = fa.bwd_varlen(qb, block(kc, src), block(vc, src), ob, lb, dob, causal=c, scale=scale)
            dq16[:, rank * blk:(rank + 1) * blk] += gq.float()
            dk16[:, src * blk:(src + 1) * blk] += gk.float()
            dv16[:, src * blk:(src + 1) * blk] += gv.float()
    torch.cuda.synchronize()
    errs, errs16 = [], []
    for got, got16, want in ((dq, dq16, rq), (dk, dk16, rk), (dv, dv16, rv)):
        errs.append(rel_fro(f64(got).transpose(0, 2, 1, 3), want))
        errs16.append(rel_fro(f64(got16).transpose(0, 2, 1, 3), want))
    # Summing fp32 shares is at least as accurate as summing bf16-rounded ones, and clearly more
    # accurate for dK, dV, the sums over the ring's key blocks (the dQ share of a row block is
    # rounded only once in both: its post-pass output).
    print(f"ring backward rel. Frobenius error, fp32 shares {errs}, bf16 shares {errs16}")
    assert all(e <= e16 * 1.02 for e, e16 in zip(errs, errs16)), (errs, errs16)
    assert errs[1] < errs16[1] and errs[2] < errs16[2], (errs, errs16)


@pytest.mark.parametrize("packed", [False, True])
def test_backward_accumulate_adds_fp32_shares(packed):
    """fa_bwd_varlen_accumulate adds its fp32 dQ, dK, dV into the caller's accumulators: starting
    from random contents, the difference after one call matches the oracle gradients, a second call
    adds the same again, and rows outside every sequence are left as they were."""
    g = torch.Generator().manual_seed(77)
    d, H, Hkv, scale = 128, 4, 2, 0.09
    if packed:
        lens = [130, 0, 257]
        cu = torch.tensor([0, 130, 130, 387], dtype=torch.int32)
        rows = 400  # 13 spare rows
        q, do = bf16((rows, H, d), g), bf16((rows, H, d), g)
        k, v = bf16((rows, Hkv, d), g), bf16((rows, Hkv, d), g)
        kw = dict(cu_seqlens_q=cu.cuda(), cu_seqlens_k=cu.cuda(), max_seqlen_q=max(lens), max_seqlen_k=max(lens))
    else:
        q, do = bf16((2, 300, H, d), g), bf16((2, 300, H, d), g)
        k, v = bf16((2, 300, Hkv, d), g), bf16((2, 300, Hkv, d), g)
        kw = {}
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.fwd_varlen(qc, kc, vc, causal=True, scale=scale, **kw)
    acc0 = [torch.randn(t.shape, generator=g).cuda() for t in (q, k, v)]
    acc = [a.clone() for a in acc0]
    fa.bwd_varlen_accumulate(qc, kc, vc, o, lse, doc, *acc, causal=True, scale=scale, **kw)
    torch.cuda.synchronize()
    one = [a - a0 for a, a0 in zip(acc, acc0)]
    if packed:
        rq, rk, rv = oracle.attention_backward_varlen(f64(q), f64(k), f64(v), f64(do), cu.numpy(), cu.numpy(), scale,
                                                      causal=True)
        for got, want in zip(one, (rq, rk, rv)):
            rel_fro(f64(got)[:387], want[:387])
            assert (got[387:] == 0).all()  # spare rows untouched
    else:
        t4 = lambda x: f64(x).transpose(0, 2, 1, 3)
        rq, rk, rv = oracle.attention_backward(t4(q), t4(k), t4(v), t4(do), scale, causal=True)
        for got, want in zip(one, (rq, rk, rv)):
            rel_fro(f64(got).transpose(0, 2, 1, 3), want)
    fa.bwd_varlen_accumulate(qc, kc, vc, o, lse, doc, *acc, causal=True, scale=scale, **kw)
    torch.cuda.synchronize()
    for a, a0, x in zip(acc, acc0, one):  # a second call adds the same shares again
        assert torch.allclose(a - a0, 2 * x, atol=1e-4, rtol=1e-4)
