"""The seeded input generator (shared by both sides; holds no method arithmetic)."""

import numpy as np
import pytest

import synth


def test_splitmix64_published_vectors():
    # First outputs of the splitmix64 generator started from state 0: the
    # output function applied to 0, 1*gamma, 2*gamma (gamma = 0x9E3779B97F4A7C15).
    g = 0x9E3779B97F4A7C15
    z = synth.splitmix64_np(np.array([0, g, (2 * g) & (2**64 - 1)], dtype=np.uint64))
    assert [hex(int(v)) for v in z] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4", "0x6c45d188009454f"]


def test_grid_values_exact_and_in_range():
    x = synth.uniform_pm1_np(synth.SEED_SCALE, 1 << 16)
    assert x.dtype == np.float32
    assert x.min() >= -1.0 and x.max() < 1.0
    k = x.astype(np.float64) * 2**23
    assert np.all(k == np.round(k)), "not on the 2**-23 grid"
    nz = np.abs(x[x != 0])
    assert nz.min() >= 2**-23, "subnormal or off-grid value"
    c = synth.coeffs_np(128)
    assert c.shape == (129,) and c.min() >= -0.5 and c.max() < 0.5


def test_offset_generation_matches_whole():
    whole = synth.uniform_pm1_np(7, 1000)
    part = synth.uniform_pm1_np(7, 300, start=500)
    assert np.array_equal(whole[500:800].view(np.uint32), part.view(np.uint32))


def test_seeds_differ():
    a = synth.uniform_pm1_np(1, 4096)
    b = synth.uniform_pm1_np(2, 4096)
    assert (a != b).mean() > 0.99


def test_torch_generator_matches_numpy_cpu():
    torch = pytest.importorskip("torch")
    for seed, n, chunk in ((synth.SEED_POLY, 5000, 1 << 26), (123, 70001, 4096)):
        t = synth.uniform_pm1_torch(seed, n, "cpu", chunk=chunk).numpy()
        assert np.array_equal(t.view(np.uint32), synth.uniform_pm1_np(seed, n).view(np.uint32))

