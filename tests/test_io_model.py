"""Pins the harness's IO / roofline model to the numbers printed on the FlashAttention plate
("FlashAttention.", Kernels and Efficiency plate 4, sections 'Workshop' and 'Never write the scores')."""

import json
import os

import pytest

from exact_io_aware_38_gb300 import roofline as rl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plate_io_model.json")


def _value(item, M, c):
    N, d = item["N"], item["d"]
    heads = c["heads"]
    std_s, fa_s = rl.plate_layer_times(N, d, heads, M, c["peak_flops"], c["bandwidth"], c["elem_bytes"])
    what = item["what"]
    if what == "bytes ratio standard / flash":
        return rl.standard_traffic_elems(N, d) / rl.flash_traffic_elems(N, d, M)
    if what == "time ratio standard / flash":
        return std_s / fa_s
    if what == "standard ms per layer":
        return std_s * 1e3
    if what == "flash ms per layer":
        return fa_s * 1e3
    if what == "score GB per layer":
        return rl.score_bytes(N, heads, c["elem_bytes"]) / 1e9
    if what == "score TB per layer":
        return rl.score_bytes(N, heads, c["elem_bytes"]) / 1e12
    raise KeyError(what)


def test_plate_numbers_reproduce():
    g = json.load(open(GOLDEN))
    M = g["model"]["M_elems"]
    for item in g["printed"]:
        got = _value(item, M, g["constants"])
        assert abs(got - item["value"]) <= item["abs_tol"], (item, got)


def test_plate_sram_reading_matters():
    # 228 000 bytes instead of 228 KiB misses the printed 11.8x: the reading is pinned, not free.
    g = json.load(open(GOLDEN))
    item = g["printed"][0]
    got = _value(item, 228000 // 2, g["constants"])
    assert abs(got - item["value"]) > item["abs_tol"]


def test_flop_convention():
    f = rl.attention_flops(1, 32, 8192, 128, causal=True)
    assert f["fwd"] == pytest.approx(4 * 32 * 8192**2 * 128 / 2)
    assert f["bwd"] == pytest.approx(2.5 * f["fwd"])
    assert f["total"] == pytest.approx(1924.145e9, rel=1e-5)
    import numpy as np

    bm = np.eye(4, dtype=np.uint8)
    f = rl.attention_flops(1, 2, 512, 64, block_mask=bm)
    assert f["fwd"] == 4 * 128 * 128 * 64 * 4 * 2


def test_tile_grid_matches_oracle():
    """The product's host tile predicate equals the oracle's 'block holds a valid pair' grid."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(5)
    for N in (1, 100, 128, 129, 300, 512):
        nb = (N + 127) // 128
        bm = (rng.random((nb, nb)) < 0.5).astype(np.uint8)
        for causal in (False, True):
            for L in (None, 1, max(1, N // 2), N):
                for mask in (None, bm):
                    a = rl.tile_visit_grid(N, causal, mask, L)
                    b = oracle.tile_grid(N, causal, mask, L)
                    assert (a == b).all(), (N, causal, L)
        if N % 128 == 0:  # whole tiles, no causal mask, no key padding: the grid is the block mask
            assert (oracle.tile_grid(N, False, bm, None) == (bm != 0)).all(), N
