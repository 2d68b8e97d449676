"""The seeded input recipes: what the module's header states about each workload holds."""

import math

import torch

from exact_io_aware_38_gb300 import workloads as W


def test_recipe_is_deterministic_and_draws_q_first():
    w = W.WORKLOADS["c3"]
    a = W.make_inputs(w, B=1, H=2, N=256)
    b = W.make_inputs(w, B=1, H=2, N=256)
    for n in ("q", "k", "v", "do"):
        assert torch.equal(a[n], b[n]) and a[n].dtype == torch.bfloat16
    c = W.make_inputs(w, B=1, H=2, N=256, seed=w.seed + 1)
    assert not torch.equal(a["q"], c["q"])
    # Q is the generator's first draw, times the workload's std, rounded to bf16
    g = torch.Generator("cpu").manual_seed(w.seed)
    q0 = (torch.randn((1, 2, 256, w.d), generator=g, dtype=torch.float32) * 3.0).to(torch.bfloat16)
    assert torch.equal(a["q"], q0)


def test_shapes_and_grouped_heads():
    for name, w in W.WORKLOADS.items():
        H = w.H // w.kv_heads * 2 if w.Hkv else 2  # a multiple of the group size
        inp = W.make_inputs(w, B=1, H=H, N=256)
        G = w.H // w.kv_heads
        assert inp["q"].shape == (1, H, 256, w.d) and inp["do"].shape == (1, H, 256, w.d)
        assert inp["k"].shape == (1, H // G, 256, w.d) and inp["v"].shape == (1, H // G, 256, w.d)
        assert inp["causal"] == w.causal and inp["scale"] == 1.0 / math.sqrt(w.d)
        assert (inp["seqlens_k"] is not None) == w.key_padding
        assert (inp["block_mask"] is not None) == w.block_sparse


def test_c2_key_lengths_uniform_on_384_to_512():
    w = W.WORKLOADS["c2"]
    inp = W.make_inputs(w, H=1)
    L = inp["seqlens_k"]
    assert L.dtype == torch.int32 and L.shape == (w.B,)
    assert int(L.min()) >= 384 and int(L.max()) <= 512
    # many draws of the same recipe cover the whole range, both ends included
    seen = set()
    for s in range(200):
        seen |= set(W.make_inputs(w, B=8, H=1, N=512, seed=s)["seqlens_k"].tolist())
    assert min(seen) == 384 and max(seen) == 512 and len(seen) > 100


def test_c3_query_and_key_std_3():
    w = W.WORKLOADS["c3"]
    inp = W.make_inputs(w, B=1, H=4, N=1024)
    for n, want in (("q", 3.0), ("k", 3.0), ("v", 1.0), ("do", 1.0)):
        s = float(inp[n].float().std())
        assert abs(s - want) < 0.03 * want, (n, s)


def test_c5_mask_band_and_density():
    w = W.WORKLOADS["c5"]
    m = W.make_inputs(w, B=1, H=1)["block_mask"]
    nb = w.nb
    assert m.dtype == torch.uint8 and m.shape == (nb, nb)
    idx = torch.arange(nb)
    assert bool((m[idx, idx] == 1).all()) and bool((m[idx[1:], idx[1:] - 1] == 1).all())
    band = torch.zeros(nb, nb, dtype=torch.bool)
    band[idx, idx] = True
    band[idx[1:], idx[1:] - 1] = True
    off = m[~band].double()
    n = off.numel()
    kept = float(off.sum())
    assert abs(kept - 0.08 * n) < 5 * math.sqrt(0.08 * 0.92 * n), (kept, n)
    assert bool((m.sum(dim=1) > 0).all())


def test_fp8_recipe_matches_the_oracle_quantiser():
    """make_fp8_inputs draws Q, K, V as make_inputs does, divides each (b, head) by max|x| / 448 and
    rounds to e4m3: the same values as the oracle's own quantiser gives, none saturated, and V
    comes back transposed."""
    import numpy as np

    from oracle import fp8

    w = W.WORKLOADS["c4"]
    inp = W.make_fp8_inputs(w, H=2)
    base = W.make_inputs(w, H=2, _keep_fp32=True)
    for n in ("q", "k", "v"):
        desc = inp[n + "_descale"]
        x = (base["_f32_" + n] / desc[:, :, None, None]).double().numpy()
        want = fp8.e4m3_quantize(x)
        got = inp[n + "8"] if n != "v" else inp["vt8"].transpose(-1, -2)
        got = got.double().numpy()
        assert np.array_equal(got, want), n
        assert np.abs(got).max() <= 448.0 and np.isclose(np.abs(got).max(), 448.0)
    a = W.make_inputs(w, H=2)
    assert all(torch.equal(a[n], base[n]) for n in ("q", "k", "v", "do"))  # the fp32 option changes no draw
