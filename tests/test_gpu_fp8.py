"""GPU parity of the FP8 forward (fa_fwd_fp8) against the fp64 oracle on the same e4m3 inputs.

The oracle is exact attention over the dequantised inputs (``oracle.fp8.attention_forward_fp8``).
Tolerances, derived from the arithmetic (see ``oracle.fp8``): the kernel's scores are exact e4m3
products summed in fp32 and its probabilities are rounded to e4m3 as 2^8 P, so per element
|O - O_ref| <= sum_j max(2^-4 P_ij, 2^-18) |v_jk| + 2^-8 |O_ref| + 1e-3 (the P rounding bound, the
bf16 output rounding with a factor 2 of margin, and fp32 noise); on average the error stays below
the root-mean-square estimate of those roundings; the LSE (from the unrounded fp32 exponentials)
stays within 1e-3 and is -inf exactly where the oracle's is. Tile visits are compared bit-exactly.
"""

import numpy as np
import pytest
import torch

import exact_io_aware_38_gb300 as fa
import oracle
from exact_io_aware_38_gb300 import build, workloads
from oracle import fp8

pytestmark = pytest.mark.gpu

LSE_MAX = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    fa.lib()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def run_gpu(inp):
    dev = "cuda"
    q8, k8, vt8 = (inp[n].to(dev) for n in ("q8", "k8", "vt8"))
    B, H, N, d = q8.shape
    nb = (N + 127) // 128
    bm = None if inp.get("block_mask") is None else inp["block_mask"].to(dev).contiguous()
    sl = None if inp.get("seqlens_k") is None else inp["seqlens_k"].to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tv = torch.full((B * H * nb,), -1, dtype=torch.int32, device=dev)
    o, lse = fa.fwd_fp8(q8, k8, vt8, *(inp[n].to(dev) for n in ("q_descale", "k_descale", "v_descale")),
                        causal=inp["causal"], block_mask=bm, seqlens_k=sl, scale=inp["scale"], tile_visits=tv,
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))
    return o.cpu(), lse.cpu(), tv.cpu().view(B, H, nb)


def deq(inp, b, h):
    """Dequantised fp64 q, k, v of query head h of sequence b."""
    H, Hkv = inp["q8"].shape[1], inp["k8"].shape[1]
    hk = oracle.kv_head(h, H, Hkv)
    q = inp["q8"][b, h].double().numpy() * float(inp["q_descale"][b, h])
    k = inp["k8"][b, hk].double().numpy() * float(inp["k_descale"][b, hk])
    v = inp["vt8"][b, hk].double().numpy().T * float(inp["v_descale"][b, hk])
    return q, k, v


def check_rows(o, lse, inp, b, h, rows):
    """O and LSE of `rows` of head (b, h) against the oracle, with the derived tolerances."""
    q, k, v = deq(inp, b, h)
    N = q.shape[0]
    bm = None if inp.get("block_mask") is None else inp["block_mask"].numpy()
    L = None if inp.get("seqlens_k") is None else int(inp["seqlens_k"][b])
    c = inp["scale"]
    om, lm = oracle.head_forward(q, k, v, c, inp["causal"], bm, L, rows=rows)
    got_o = o[b, h][rows].double().numpy()
    got_l = lse[b, h][rows].double().numpy()
    empty = np.isneginf(lm)
    assert (np.isneginf(got_l) == empty).all()
    if (~empty).any():
        assert np.abs(got_l[~empty] - lm[~empty]).max() <= LSE_MAX
    assert (got_o[empty] == 0).all()
    # exact probabilities of these rows, for the error bound
    valid = oracle.valid_matrix(rows, N, inp["causal"], bm, L)
    with np.errstate(over="ignore", invalid="ignore"):
        p = np.where(valid, np.exp(c * (q[rows] @ k.T) - np.where(empty, 0.0, lm)[:, None]), 0.0)
    err = np.abs(got_o - om)
    bound = fp8.p_rounding_bound(p, np.abs(v)) + 2.0 ** -8 * np.abs(om) + 1e-3
    assert (err <= bound).all(), (b, h, float((err - bound).max()))
    rms = np.sqrt(fp8.p_rounding_rms(p, v) ** 2 + (2.0 ** -9 * np.abs(om)) ** 2 / 3.0)
    assert err.mean() <= rms.mean() + 1e-4, (b, h, err.mean(), rms.mean())
    return err


def check_visits(tv, inp):
    B, H, N, _ = inp["q8"].shape
    bm = None if inp.get("block_mask") is None else inp["block_mask"].numpy()
    for b in range(B):
        L = None if inp.get("seqlens_k") is None else int(inp["seqlens_k"][b])
        want = oracle.tile_grid(N, inp["causal"], bm, L).sum(axis=1)
        for h in range(H):
            assert (tv[b, h].numpy() == want).all(), (b, h)


def small_fp8_inputs(B, H, Hkv, N, kind, seed):
    w = workloads.Workload("t", B, H, N, 128, causal="causal" in kind, seed=seed, Hkv=Hkv)
    inp = workloads.make_fp8_inputs(w)
    g = torch.Generator().manual_seed(seed + 7)
    nb = (N + 127) // 128
    if "pad" in kind:
        inp["seqlens_k"] = torch.randint(1, N + 1, (B,), generator=g, dtype=torch.int32)
    if "block" in kind:
        inp["block_mask"] = (torch.rand((nb, nb), generator=g) < 0.5).to(torch.uint8)
        inp["block_mask"][torch.arange(nb), torch.arange(nb)] = 1
    return inp


@pytest.mark.parametrize("N", [128, 256, 384, 1040])
@pytest.mark.parametrize("kind", ["dense", "causal", "pad", "block", "causal+pad+block"])
@pytest.mark.parametrize("Hkv", [4, 2])
def test_fp8_small_parity(N, kind, Hkv):
    inp = small_fp8_inputs(2, 4, Hkv, N, kind, seed=N + len(kind) * 31 + Hkv)
    o, lse, tv = run_gpu(inp)
    for b in range(2):
        for h in range(4):
            check_rows(o, lse, inp, b, h, np.arange(N))
    check_visits(tv, inp)


def test_fp8_long_context_every_head_sampled():
    """The long-context causal shape (B1 H32 N8192 d128) at full size: 128 sampled rows of every
    head against the oracle, tile visits of every head, finite outputs."""
    inp = workloads.make_fp8_inputs(workloads.WORKLOADS["c4"])
    o, lse, tv = run_gpu(inp)
    assert torch.isfinite(o.float()).all()
    rng = np.random.default_rng(41)
    worst = 0.0
    for h in range(inp["q8"].shape[1]):
        rows = np.sort(rng.choice(8192, 128, replace=False))
        worst = max(worst, float(check_rows(o, lse, inp, 0, h, rows).max()))
    check_visits(tv, inp)
    assert worst > 0  # the comparison is not trivially exact
