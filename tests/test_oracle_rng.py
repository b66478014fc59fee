"""Pins for the oracle's SplitMix64 table generator."""
import numpy as np
from scipy import stats

from oracle import rng
from conftest import golden

M64 = (1 << 64) - 1


def _sequential(state, n):
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_published_outputs_from_state_zero():
    g = golden("splitmix64_seed0.json")
    want = [int(h, 16) for h in g["outputs_hex"]]
    got = [int(x) for x in rng.words(0, 0, len(want))]
    assert got == want


def test_counter_form_equals_sequential_generator():
    for seed, stream in [(0, 1), (7, 2), (123456789, 1), (2**40 - 1, 2)]:
        s0 = (seed + stream * (1 << 40)) & M64
        assert [int(x) for x in rng.words(seed, stream, 50)] == _sequential(s0, 50)


def test_signs_balanced_and_pm_one():
    s = rng.signs(0, 1 << 16)
    assert set(np.unique(s)) == {-1.0, 1.0}
    assert abs(s.mean()) < 4.0 / np.sqrt(s.size)


def test_gaussian_matrix_is_standard_normal():
    s = rng.gaussian_matrix(1, 512, 512).astype(np.float64).ravel()
    assert s.dtype == np.float64
    assert abs(s.mean()) < 5.0 / np.sqrt(s.size)
    assert abs(s.var() - 1.0) < 0.02
    assert stats.kstest(s, "norm").pvalue > 1e-3


def test_box_muller_pairs():
    """S_flat[2k], S_flat[2k+1] are the cos/sin pair built from words 2k, 2k+1."""
    w = [int(x) for x in rng.words(5, 2, 4)]
    u1 = ((w[0] >> 11) + 1) * 2.0 ** -53
    u2 = (w[1] >> 11) * 2.0 ** -53
    r = np.sqrt(-2 * np.log(u1))
    s = rng.gaussian_matrix(5, 1, 4).ravel()
    assert s[0] == np.float32(r * np.cos(2 * np.pi * u2))
    assert s[1] == np.float32(r * np.sin(2 * np.pi * u2))
