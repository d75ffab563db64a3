"""The seeded generators: determinism, independent slices, distribution recipe."""

import numpy as np

from workloads import configs, rng


def test_splitmix64_reference_values():
    """Counter mode from key 0 reproduces SplitMix64's published first outputs for seed 0."""
    out = rng._mix(np.array([0x9E3779B97F4A7C15, 0x3C6EF372FE94F82A], dtype=np.uint64))
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_slices_equal_full_batch():
    w = configs.config1(batch=8)
    full = w.step(3)
    part = w.step(3, 5, 7)
    for k in full:
        assert np.array_equal(full[k][5:7], part[k])
    assert np.array_equal(w.S0()[2:4], w.S0(2, 4))
    g = configs.config2(batch=6)
    assert np.array_equal(g.draft(1, 4)["k"][1:3], g.draft(1, 4, 1, 3)["k"])


def test_determinism_and_stream_separation():
    a = configs.config1(batch=4).step(0)
    b = configs.config1(batch=4).step(0)
    c = configs.config1(batch=4).step(1)
    assert all(np.array_equal(a[k], b[k]) for k in a)
    assert not np.array_equal(a["x"], c["x"])


def test_distribution_recipe():
    w = configs.config1(batch=16)
    d = {k: rng.bf16_bits_to_float(v) for k, v in w.step(0).items()}
    assert abs(d["x"].std() - 1.0) < 0.02
    assert abs(d["B"].std() * np.sqrt(128) - 1.0) < 0.05
    assert d["dt"].min() > 0
    A = w.A()
    assert np.all(A <= -1.0) and np.all(A >= -8.0)
    g = configs.config2(batch=4).step(0)
    qn = np.linalg.norm(rng.bf16_bits_to_float(g["q"]), axis=-1)
    assert np.allclose(qn, 1.0, atol=1e-2)
    assert np.all((g["beta"] > 0) & (g["beta"] < 1)) and np.all(g["g"] <= 0)


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], dtype=np.float32)
    bits = rng.float32_to_bf16_bits(x)
    assert rng.bf16_bits_to_float(bits).tolist() == [1.0, 1.015625, -2.5]


def test_accepted_counts_uniform():
    acc = configs.config3_mamba2().accepted(0, 4)
    assert acc.min() == 0 and acc.max() == 4
    assert abs(acc.mean() - 2.0) < 0.25
