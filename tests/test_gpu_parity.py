"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Tolerances (bf16 inputs/outputs, fp32 accumulation): O max-abs <= 2e-2 and mean-abs <= 2e-3;
LSE max-abs <= 1e-3 (and -inf exactly where a row has no valid key); dQ, dK, dV relative
Frobenius error <= 2e-2 each. Tile-skip decisions of both passes are compared bit-exactly with the
oracle's "block holds a valid pair" grid: the forward's key tiles per query tile, and the backward's
64-row query steps per key tile.
"""

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


def run_gpu(inp, backward=True, visits=False):
    dev = "cuda"
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    B, H, N, d = q.shape
    nb = (N + 127) // 128
    bm = None if inp.get("block_mask") is None else inp["block_mask"].to(dev).contiguous()
    sl = None if inp.get("seqlens_k") is None else inp["seqlens_k"].to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tv = torch.full((B * H * nb,), -1, dtype=torch.int32, device=dev) if visits else None
    Hkv = k.shape[1]
    sv = torch.full((B * Hkv * nb,), -1, dtype=torch.int32, device=dev) if visits and backward else None
    kw = dict(causal=inp["causal"], block_mask=bm, seqlens_k=sl, scale=inp["scale"], status=status)
    o, lse = fa.fwd(q, k, v, tile_visits=tv, **kw)
    out = {"o": o, "lse": lse}
    if backward:
        out["dq"], out["dk"], out["dv"] = fa.bwd(q, k, v, o, lse, do, step_visits=sv, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))
    res = {n: t.cpu() for n, t in out.items()}
    if visits:
        res["visits"] = tv.cpu().view(B, H, nb)
    if sv is not None:
        res["step_visits"] = sv.cpu().view(B, Hkv, nb)
    return res


def f64(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, dtype=np.float64)


def check_o_lse(o, lse, o_ref, lse_ref):
    o, lse = f64(o), f64(lse)
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    empty = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == empty).all()
    if (~empty).any():
        assert np.abs(lse[~empty] - lse_ref[~empty]).max() <= LSE_MAX
    assert (o[empty.reshape(o.shape[:-1])] == 0).all()


def rel_fro(x, ref):
    x, ref = f64(x), np.asarray(ref)
    nr = np.linalg.norm(ref)
    if nr == 0:
        # An analytically zero gradient (e.g. N = 1 or a single valid key: dS = P (dP - D) cancels)
        # leaves only rounding noise, since the kernel's D uses the stored bf16 O.
        assert np.abs(x).max() <= 1e-3
        return 0.0
    r = np.linalg.norm(x - ref) / nr
    assert r <= REL_FRO, r
    return r


def oracle_args(inp):
    bm = None if inp.get("block_mask") is None else inp["block_mask"].numpy()
    sl = None if inp.get("seqlens_k") is None else inp["seqlens_k"].numpy()
    return dict(causal=inp["causal"], block_mask=bm, seqlens_k=sl)


def full_check(inp, backward=True):
    got = run_gpu(inp, backward=backward, visits=True)
    ref_o, ref_lse = oracle.attention_forward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), inp["scale"], **oracle_args(inp))
    check_o_lse(got["o"], got["lse"], ref_o, ref_lse)
    if backward:
        g = oracle.attention_backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["do"]), inp["scale"],
                                      **oracle_args(inp))
        for name, ref in zip(("dq", "dk", "dv"), g):
            rel_fro(got[name], ref)
    check_visits(got, inp)
    return got


def check_visits(got, inp):
    """Forward: key tiles visited per (b, h, query tile) = row sums of the oracle's grid. Backward:
    64-row query steps visited per (b, K/V head, key tile) = the steps of the query tiles in the
    grid's column (a tile of rows 128 I .. has the steps 2 I and, if row 64 (2 I + 1) exists,
    2 I + 1), times the query heads sharing the K/V head."""
    B, H, N, _ = inp["q"].shape
    Hkv = inp["k"].shape[1]
    a = oracle_args(inp)
    nb = (N + 127) // 128
    steps_in = np.array([1 + int((2 * i + 1) * 64 < N) for i in range(nb)])
    for b in range(B):
        L = None if a["seqlens_k"] is None else int(a["seqlens_k"][b])
        grid = oracle.tile_grid(N, a["causal"], a["block_mask"], L)
        want = grid.sum(axis=1)
        for h in range(H):
            assert (got["visits"][b, h].numpy() == want).all(), (b, h)
        if "step_visits" in got:
            want_b = (H // Hkv) * (grid * steps_in[:, None]).sum(axis=0)
            for hk in range(Hkv):
                assert (got["step_visits"][b, hk].numpy() == want_b).all(), (b, hk)


def small_inputs(B, H, N, d, kind, seed):
    inp = workloads.random_inputs(B, H, N, d, seed)
    inp.update(causal=False, block_mask=None, seqlens_k=None, scale=1.0 / np.sqrt(d))
    g = torch.Generator().manual_seed(seed + 7)
    nb = (N + 127) // 128
    if "causal" in kind:
        inp["causal"] = True
    if "pad" in kind:
        inp["seqlens_k"] = torch.randint(1, N + 1, (B,), generator=g, dtype=torch.int32)
    if "block" in kind:
        inp["block_mask"] = (torch.rand((nb, nb), generator=g) < 0.5).to(torch.uint8)
        inp["block_mask"][torch.arange(nb), torch.arange(nb)] = 1
    return inp


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 256, 300, 384])
@pytest.mark.parametrize("kind", ["dense", "causal", "pad", "block", "causal+pad+block"])
def test_small_parity(N, d, kind):
    full_check(small_inputs(2, 3, N, d, kind, seed=N * 10 + d))


def test_degenerate_masks():
    """Rows with no valid key (a block row of zeros, a zero key length) give O = 0, LSE = -inf,
    dQ = 0; masked keys get dK = dV = 0."""
    B, H, N, d = 2, 2, 384, 64
    inp = workloads.random_inputs(B, H, N, d, 77)
    bm = torch.ones((3, 3), dtype=torch.uint8)
    bm[1, :] = 0
    inp.update(causal=True, block_mask=bm, seqlens_k=torch.tensor([0, 200], dtype=torch.int32), scale=0.125)
    got = full_check(inp)
    assert (got["dq"][0] == 0).all() and (got["dk"][0] == 0).all() and (got["dv"][0] == 0).all()
    assert (got["dk"][1, :, 200:] == 0).all()
    assert torch.isneginf(got["lse"][:, :, 128:256]).all()


def test_host_mask_arrays_are_rejected():
    """A block mask or key lengths in plain host memory would fault the kernel: the library checks
    where they live before any launch and returns FA_ERR_INVALID_ARG; a device copy runs."""
    B, H, N, d = 1, 2, 256, 64
    g = torch.Generator().manual_seed(1)
    q, k, v = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    host_mask = np.ones(4, dtype=np.uint8)
    host_len = np.array([100], dtype=np.int32)
    stream = torch.cuda.current_stream().cuda_stream
    call = lambda bm, sl: fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                                    0, bm, sl, 0.125, None, None, stream)
    assert call(host_mask.ctypes.data, None) == -1
    assert call(None, host_len.ctypes.data) == -1
    dev_mask = torch.from_numpy(host_mask).cuda()
    assert call(dev_mask.data_ptr(), None) == 0
    torch.cuda.synchronize()


def test_block_mask_rows_longer_than_the_bitmap():
    """Block-sparse rows of 2051 key tiles, more than the 2048 the forward's per-CTA bitmap covers
    (the rest are looked up tile by tile), and as many query tiles: O and LSE on sampled rows
    against the oracle, and every skip decision of both passes bit-exactly. With no causal mask, no
    key padding and whole tiles, the oracle's visit grid is the block mask itself (pinned against
    oracle.tile_grid on small sizes in test_io_model); its brute force is too slow at this size."""
    nb = 2051
    B, H, N, d = 1, 1, nb * 128, 64
    inp = workloads.random_inputs(B, H, N, d, 11)
    rng = np.random.default_rng(12)
    bm = (rng.random((nb, nb)) < 0.01).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    bm[:, nb - 3:] = 1  # every row also sees the key tiles past the bitmap's reach
    inp.update(causal=False, block_mask=torch.from_numpy(bm), seqlens_k=None, scale=0.125)
    got = run_gpu(inp, backward=True, visits=True)
    rows = np.sort(rng.choice(N, 64, replace=False))
    om, lm = oracle.head_forward(f64(inp["q"][0, 0]), f64(inp["k"][0, 0]), f64(inp["v"][0, 0]), 0.125, False, bm,
                                 None, rows=rows)
    check_o_lse(got["o"][0, 0][rows], got["lse"][0, 0][rows], om, lm)
    grid = bm != 0
    assert (got["visits"][0, 0].numpy() == grid.sum(axis=1)).all()
    assert (got["step_visits"][0, 0].numpy() == 2 * grid.sum(axis=0)).all()  # two 64-row steps per tile
    for n in ("o", "dq", "dk", "dv"):
        assert torch.isfinite(got[n].float()).all(), n


@pytest.mark.parametrize("d", [64, 128])
def test_all_tiles_masked(d):
    """Every key tile has no visited step: each is taken from the queue, skipped by the issuers,
    and its dK/dV rows are written as zeros."""
    inp = workloads.random_inputs(1, 2, 256, d, 5)
    inp.update(causal=False, block_mask=torch.zeros((2, 2), dtype=torch.uint8), seqlens_k=None, scale=0.1)
    got = full_check(inp)
    assert (got["visits"] == 0).all() and (got["step_visits"] == 0).all()
    assert (got["dk"] == 0).all() and (got["dv"] == 0).all()


@pytest.mark.parametrize("d", [64, 128])
def test_empty_key_tile_columns(d):
    """Key tiles whose block-mask column is empty (no query tile sees them) between ones that are
    seen, with a causal mask and a short last tile: the empty tiles' dK/dV are zero, the rest match
    the oracle, and every skip decision matches bit-exactly."""
    B, H, N = 2, 2, 5 * 128 + 40
    inp = workloads.random_inputs(B, H, N, d, 91)
    nb = (N + 127) // 128
    bm = torch.ones((nb, nb), dtype=torch.uint8)
    bm[:, 1] = 0
    bm[:, 3] = 0
    bm[0, 3] = 1  # column 3 is seen only by query tile 0, which the causal mask then hides
    inp.update(causal=True, block_mask=bm, seqlens_k=None, scale=1.0 / np.sqrt(d))
    got = full_check(inp)
    for kt in (1, 3):
        assert (got["dk"][:, :, kt * 128:(kt + 1) * 128] == 0).all(), kt
        assert (got["dv"][:, :, kt * 128:(kt + 1) * 128] == 0).all(), kt
        assert (got["step_visits"][:, :, kt] == 0).all(), kt


def test_repeatable():
    inp = small_inputs(2, 4, 640, 128, "causal", 3)
    a = run_gpu(inp)
    b = run_gpu(inp)
    for n in ("o", "lse", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n
    assert (a["dq"].float() - b["dq"].float()).abs().max() <= 1e-2


@pytest.mark.parametrize("d", [64, 128])
def test_back_to_back_calls_reuse_buffers(d):
    """The kernels run as programmatic dependents of the kernel before them on the stream. Calls
    queued back to back, with no host synchronisation, that reuse the same O, LSE, gradient and
    workspace buffers (each call's pre pass clears the accumulator the previous call's post pass
    reads; each forward overwrites the O and LSE the previous backward read) must give the results
    of the same calls made one at a time."""
    dev = "cuda"
    inputs = [small_inputs(2, 4, 640, d, "causal", 11), small_inputs(2, 4, 640, d, "causal", 12)]
    dev_in = [{n: inp[n].to(dev) for n in ("q", "k", "v", "do")} for inp in inputs]
    shape = dev_in[0]["q"]
    o, lse = torch.empty_like(shape), torch.empty((2, 4, 640), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(shape), torch.empty_like(shape), torch.empty_like(shape)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(2, 4, 640, d), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    snaps = []
    for t in (dev_in[0], dev_in[1], dev_in[0], dev_in[1]):
        fa.fwd(t["q"], t["k"], t["v"], causal=True, out=o, lse=lse, status=status)
        fa.bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=True, dq=dq, dk=dk, dv=dv, workspace=ws, status=status)
        snaps.append([x.clone() for x in (o, lse, dq, dk, dv)])  # stream-ordered copies, no host sync
    snaps = [[x.cpu() for x in snap] for snap in snaps]
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i, inp in enumerate(inputs):
        ref = run_gpu(inp)  # the same call alone, fresh buffers
        for got in (snaps[i], snaps[i + 2]):
            for n, x in zip(("o", "lse", "dk", "dv"), (got[0], got[1], got[3], got[4])):
                assert torch.equal(x, ref[n]), n
            # dQ is summed with fp32 reduce-adds in no fixed order
            assert (got[2].float() - ref["dq"].float()).abs().max() <= 1e-2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (8, 1), (6, 3), (4, 4)])
@pytest.mark.parametrize("N,kind", [(129, "dense"), (300, "causal"), (384, "causal+pad+block")])
def test_gqa_parity(H, Hkv, N, kind, d):
    """Grouped-query attention: K/V heads shared by H / Hkv query heads; dK, dV summed per group."""
    inp = small_inputs(2, H, N, d, kind, seed=N * 7 + H * 3 + Hkv + d)
    inp["k"] = inp["k"][:, :Hkv].contiguous()
    inp["v"] = inp["v"][:, :Hkv].contiguous()
    got = full_check(inp)
    assert got["dk"].shape == inp["k"].shape and got["dv"].shape == inp["v"].shape


def test_gqa_repeatable():
    """dK and dV of shared heads are summed in one CTA's tensor memory: identical bits per run."""
    inp = small_inputs(1, 8, 640, 128, "causal", 11)
    inp["k"] = inp["k"][:, :2].contiguous()
    inp["v"] = inp["v"][:, :2].contiguous()
    a = run_gpu(inp)
    b = run_gpu(inp)
    for n in ("o", "lse", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_config_full(name):
    w = workloads.WORKLOADS[name]
    full_check(workloads.make_inputs(w), backward=w.backward)


def sampled_check(inp, heads, n_rows, n_cols, seed, fwd_rows=128):
    """Full-size launch; the oracle evaluates O and LSE on `fwd_rows` sampled rows of every head,
    and sampled K/V heads (b, hk), with the query heads that share each, on sampled rows and key
    columns one by one for the gradients."""
    got = run_gpu(inp, backward=True, visits=True)
    B, H, N, d = inp["q"].shape
    Hkv = inp["k"].shape[1]
    a = oracle_args(inp)
    c = inp["scale"]
    rng = np.random.default_rng(seed)
    for b in range(B):
        L = None if a["seqlens_k"] is None else int(a["seqlens_k"][b])
        for h in range(H):
            hk = oracle.kv_head(h, H, Hkv)
            rows = np.sort(rng.choice(N, fwd_rows, replace=False))
            om, lm = oracle.head_forward(f64(inp["q"][b, h]), f64(inp["k"][b, hk]), f64(inp["v"][b, hk]), c,
                                         a["causal"], a["block_mask"], L, rows=rows)
            check_o_lse(got["o"][b, h][rows], got["lse"][b, h][rows], om, lm)
    for (b, hk) in heads:
        k, v = (f64(inp[n][b, hk]) for n in ("k", "v"))
        L = None if a["seqlens_k"] is None else int(a["seqlens_k"][b])
        cols = np.sort(rng.choice(N, n_cols, replace=False))
        dk = np.zeros((n_cols, d))
        dv = np.zeros((n_cols, d))
        for h in [h for h in range(H) if oracle.kv_head(h, H, Hkv) == hk]:
            q, do = (f64(inp[n][b, h]) for n in ("q", "do"))
            rows = np.sort(rng.choice(N, n_rows, replace=False))
            om, lm = oracle.head_forward(q, k, v, c, a["causal"], a["block_mask"], L, rows=rows)
            check_o_lse(got["o"][b, h][rows], got["lse"][b, h][rows], om, lm)
            stats = oracle.head_row_stats(q, k, v, do, c, a["causal"], a["block_mask"], L)
            dq = oracle.head_dq(q, k, v, do, c, a["causal"], a["block_mask"], L, rows=rows)
            rel_fro(got["dq"][b, h][rows], dq)
            dkh, dvh = oracle.head_dkdv(q, k, v, do, c, a["causal"], a["block_mask"], L, cols=cols, stats=stats)
            dk += dkh
            dv += dvh
        rel_fro(got["dk"][b, hk][cols], dk)
        rel_fro(got["dv"][b, hk][cols], dv)
    # Properties at full size, every head: finite outputs; sum_j dK_j = 0 (rows of dS sum to 0).
    for n in ("o", "dq", "dk", "dv"):
        assert torch.isfinite(got[n].float()).all(), n
    dk = got["dk"].double()
    colsum = dk.sum(dim=2).norm(dim=-1)
    assert (colsum <= 0.05 * dk.norm(dim=(2, 3)) + 1e-3).all()
    check_visits(got, inp)


def test_config_c4_sampled():
    inp = workloads.make_inputs(workloads.WORKLOADS["c4"])
    sampled_check(inp, heads=[(0, 0), (0, 31)], n_rows=384, n_cols=384, seed=4)


def test_config_c4g_sampled():
    """The long-context causal shape with 8 K/V heads, each shared by 4 query heads."""
    inp = workloads.make_inputs(workloads.WORKLOADS["c4g"])
    sampled_check(inp, heads=[(0, 0), (0, 7)], n_rows=256, n_cols=384, seed=6)


def test_config_c5_sampled():
    inp = workloads.make_inputs(workloads.WORKLOADS["c5"])
    sampled_check(inp, heads=[(0, 9)], n_rows=384, n_cols=384, seed=5)
