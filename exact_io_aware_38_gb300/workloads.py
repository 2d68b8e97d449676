"""Seeded synthetic attention workloads.

This module only draws inputs; it holds none of the attention arithmetic. Both the CUDA path's
tests/benchmark and the CPU oracle are fed from it.

Recipe (the same for every workload):
  * one ``torch.Generator('cpu')`` seeded with the workload's seed;
  * draw order: Q, K, V, dO (each fp32 N(0, 1) of shape [B, H, N, d], times the workload's std),
    then the key lengths or the block mask;
  * each tensor is rounded to bf16 (round-to-nearest-even) on the host. The same host bits go to
    the GPU and (upcast exactly) to the oracle.

Workloads (shapes from the five benchmark configurations; seeds 1000 + index):
  c1  B1 H1  N128   d64   no mask, forward only                         (correctness)
  c2  B8 H16 N512   d64   key padding, L_b uniform on the integers [384, 512]   (BERT-large shape)
  c3  B8 H12 N1024  d64   causal, Q and K drawn with std 3                 (GPT-2 shape)
  c4  B1 H32 N8192  d128  causal                                          (long context, headline)
  c5  B1 H16 N16384 d64   128x128 block mask: band {(I, I), (I, I-1)} plus every other block
                          kept independently with probability 0.08 (u < 0.08, u uniform, drawn
                          over the whole grid in row-major order)
Grouped-query variant (K and V drawn with Hkv heads, [B, Hkv, N, d]; seed 1006):
  c4g B1 H32 Hkv8 N8192 d128 causal   (c4's shape with four query heads per K/V head)
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

TILE = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool = False
    key_padding: bool = False
    block_sparse: bool = False
    backward: bool = True
    qk_std: float = 1.0
    seed: int = 1000
    Hkv: int | None = None  # K/V heads (grouped-query attention); None = H
    note: str = field(default="", compare=False)

    @property
    def kv_heads(self) -> int:
        return self.H if self.Hkv is None else self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def nb(self) -> int:
        return (self.N + TILE - 1) // TILE


WORKLOADS = {
    "c1": Workload("c1", 1, 1, 128, 64, backward=False, seed=1001, note="correctness, forward only"),
    "c2": Workload("c2", 8, 16, 512, 64, key_padding=True, seed=1002, note="BERT-large shape, key padding"),
    "c3": Workload("c3", 8, 12, 1024, 64, causal=True, qk_std=3.0, seed=1003, note="GPT-2 shape, causal, Q/K std 3"),
    "c4": Workload("c4", 1, 32, 8192, 128, causal=True, seed=1004, note="long-context causal (headline)"),
    "c5": Workload("c5", 1, 16, 16384, 64, block_sparse=True, seed=1005, note="block-sparse, band + 8% random"),
    "c4g": Workload("c4g", 1, 32, 8192, 128, causal=True, seed=1006, Hkv=8,
                    note="long-context causal, grouped-query (8 K/V heads)"),
}


def band_random_block_mask(nb: int, gen: torch.Generator, p: float = 0.08) -> torch.Tensor:
    """uint8 [nb, nb]: blocks (I, I) and (I, I-1) kept, every other block kept when u_IJ < p."""
    u = torch.rand((nb, nb), generator=gen, dtype=torch.float32)
    m = (u < p).to(torch.uint8)
    idx = torch.arange(nb)
    m[idx, idx] = 1
    m[idx[1:], idx[1:] - 1] = 1
    assert bool((m.sum(dim=1) > 0).all())
    return m


def make_inputs(w: Workload, *, B: int | None = None, H: int | None = None, N: int | None = None,
                seed: int | None = None, _keep_fp32: bool = False) -> dict:
    """Host (CPU) tensors for workload ``w``; B, H, N and seed may be overridden (smaller tests).

    Returns dict with q, do (bf16 [B,H,N,d]), k, v (bf16 [B,Hkv,N,d]), seqlens_k (int32 [B] or
    None), block_mask (uint8 [nb, nb] or None), causal, scale. An H override keeps H / Hkv.
    (_keep_fp32 also returns the fp32 draws as _f32_q, _f32_k, _f32_v, _f32_do.)
    """
    G = w.H // w.kv_heads
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    if H % G:
        raise ValueError(f"H={H} is not a multiple of the workload's group size {G}")
    g = torch.Generator("cpu").manual_seed(w.seed if seed is None else seed)

    f32 = {}

    def draw(name, std, heads):
        x = torch.randn((B, heads, N, w.d), generator=g, dtype=torch.float32) * std
        if _keep_fp32:
            f32["_f32_" + name] = x
        return x.to(torch.bfloat16)

    q = draw("q", w.qk_std, H)
    k = draw("k", w.qk_std, H // G)
    v = draw("v", 1.0, H // G)
    do = draw("do", 1.0, H)
    seqlens = None
    mask = None
    if w.key_padding:
        lo = min(384, N)
        seqlens = torch.randint(lo, N + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    if w.block_sparse:
        mask = band_random_block_mask((N + TILE - 1) // TILE, g)
    return dict(q=q, k=k, v=v, do=do, seqlens_k=seqlens, block_mask=mask, causal=w.causal, scale=w.scale, **f32)


def random_inputs(B, H, N, d, seed, *, std=1.0, dtype=torch.bfloat16) -> dict:
    """Plain seeded N(0, std) Q, K, V, dO for ad-hoc test shapes (same draw order as above)."""
    g = torch.Generator("cpu").manual_seed(seed)
    shape = (B, H, N, d)
    out = {}
    for name in ("q", "k", "v", "do"):
        out[name] = (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dtype)
    return out


def make_fp8_inputs(w: Workload, H: int | None = None, seed: int | None = None) -> dict:
    """e4m3 inputs for the FP8 forward with the workload's shape, masks and seed: Q, K, V are drawn
    exactly as in ``make_inputs`` (fp32 N(0,1) times the workload's std, same generator order), then
    each (b, head) slice is divided by its descale factor max|x| / 448 and converted to e4m3
    (torch's float8_e4m3fn: nearest, ties to even; nothing exceeds 448). V is returned transposed,
    [B, Hkv, d, N]. Returns q8, k8, vt8, the fp32 descales [B, H] / [B, Hkv] and the masks."""
    base = make_inputs(w, H=H, seed=seed, _keep_fp32=True)
    out = {n: base[n] for n in ("block_mask", "seqlens_k", "causal", "scale")}
    for n in ("q", "k", "v"):
        x = base["_f32_" + n]
        amax = x.abs().amax(dim=(2, 3)).clamp_min(1e-30)
        desc = (amax / 448.0).to(torch.float32)
        x8 = (x / desc[:, :, None, None]).to(torch.float8_e4m3fn)
        out[n + "_descale"] = desc
        out[n + "8"] = x8 if n != "v" else x8.transpose(-1, -2).contiguous()
    out["vt8"] = out.pop("v8")
    return out
