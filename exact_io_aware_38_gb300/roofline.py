"""FLOP, byte and roofline arithmetic for the attention kernels.

* FLOP convention (the benchmark's metric): forward = 4 B H N^2 d (two N x N x d products), backward
  = 2.5 x forward, halved exactly under a causal mask; under a block mask only the 128 x 128 tiles
  that are actually visited count, 4 * 128 * 128 * d each (forward).
* IO model of the FlashAttention plate ("FlashAttention.", Kernels and Efficiency plate 4, section
  "Workshop"): per head and forward pass, standard attention moves 4Nd + 4N^2 bf16 elements and
  FlashAttention 4Nd + 2 N^2 d^2 / M, with M the on-chip SRAM in elements; time by the roofline is
  max(flops / peak, bytes / bandwidth).
"""

from __future__ import annotations

import numpy as np

TILE = 128


def tile_visit_grid(N: int, causal: bool, block_mask=None, key_len: int | None = None) -> np.ndarray:
    """bool [nb, nb]: the (query tile, key tile) pairs the kernels visit for one head.

    Tile (I, J) is visited iff the block mask keeps it, J <= I under a causal mask, and
    J * 128 < key_len under key padding. (Every such tile holds at least one unmasked pair.)
    """
    nb = (N + TILE - 1) // TILE
    I = np.arange(nb)[:, None]
    J = np.arange(nb)[None, :]
    g = np.ones((nb, nb), dtype=bool)
    if causal:
        g &= J <= I
    if key_len is not None:
        g &= J * TILE < int(key_len)
    if block_mask is not None:
        g &= np.asarray(block_mask) != 0
    return g


def attention_flops(B, H, N, d, *, causal=False, block_mask=None, backward=True) -> dict:
    """FLOPs by the benchmark's convention: {'fwd', 'bwd', 'total'}."""
    if block_mask is not None:
        tiles = int(tile_visit_grid(N, causal, block_mask).sum())
        fwd = 4.0 * TILE * TILE * d * tiles * B * H
    else:
        fwd = 4.0 * B * H * N * N * d
        if causal:
            fwd /= 2.0
    bwd = 2.5 * fwd if backward else 0.0
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd}


def useful_padding_flops(H, N, d, seqlens) -> float:
    """Secondary forward count under key padding: 4 H d N sum_b L_b."""
    return 4.0 * H * d * N * float(np.sum(np.asarray(seqlens, dtype=np.float64)))


def algorithmic_bytes(B, H, N, d) -> dict:
    """Compulsory HBM traffic: forward reads Q, K, V and writes O (bf16) and LSE (fp32); the
    backward pass reads Q, K, V, O, dO, LSE and writes dQ, dK, dV (bf16) plus D (fp32)."""
    t = B * H * N * d * 2
    rows = B * H * N * 4
    return {"fwd": 4 * t + rows, "bwd": 8 * t + 2 * rows}


# --------------------------------------------------------------- plate's IO model ("Workshop")


def standard_traffic_elems(N, d):
    return 4 * N * d + 4 * N * N


def flash_traffic_elems(N, d, M):
    return 4 * N * d + 2 * N * N * d * d / M


def roofline_time_s(flops, nbytes, peak_flops, bandwidth):
    return max(flops / peak_flops, nbytes / bandwidth)


def plate_layer_times(N, d, heads, M, peak_flops, bandwidth, elem_bytes=2):
    """(standard seconds, flash seconds) per layer of ``heads`` heads, forward pass."""
    flops = 4.0 * N * N * d * heads
    std = roofline_time_s(flops, standard_traffic_elems(N, d) * elem_bytes * heads, peak_flops, bandwidth)
    fa = roofline_time_s(flops, flash_traffic_elems(N, d, M) * elem_bytes * heads, peak_flops, bandwidth)
    return std, fa


def score_bytes(N, heads, elem_bytes=2):
    """Memory of the N x N score matrices of one layer."""
    return N * N * elem_bytes * heads
