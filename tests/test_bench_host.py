"""Host-side arithmetic of bench.py that needs no GPU."""

from types import SimpleNamespace


def test_useful_padding_figure():
    import bench

    dense = SimpleNamespace(causal=False)
    # C2's shape with two sequences: 4 H d N sum_b L_b per forward, x3.5 with the backward, per ms.
    got = bench.useful_padding(dense, [384, 512], 16, 512, 64, 1.0, 1)
    want = 3.5 * 4 * 16 * 64 * 512 * (384 + 512) / 1e-3 / 1e12
    assert abs(got["value"] - want) <= 1e-12 * want
    assert got["unit"] == "TFLOP/s"
    # Whole-job value scales with the number of replicas.
    assert abs(bench.useful_padding(dense, [384, 512], 16, 512, 64, 1.0, 4)["value"] - 4 * want) <= 1e-12 * want
    # No key padding, or a causal mask: no secondary figure.
    assert bench.useful_padding(dense, None, 16, 512, 64, 1.0, 1) is None
    assert bench.useful_padding(SimpleNamespace(causal=True), [384], 16, 512, 64, 1.0, 1) is None


def test_step_percentiles_nearest_rank():
    import bench

    xs = [float(i) for i in range(1, 21)]  # 20 steps, 1 .. 20 ms, shuffled order must not matter
    assert bench.percentiles(list(reversed(xs))) == [2.0, 10.0, 18.0]
    assert bench.percentiles([5.0]) == [5.0, 5.0, 5.0]
    assert bench.percentiles([3.0, 1.0, 2.0], qs=(0, 100)) == [1.0, 3.0]
