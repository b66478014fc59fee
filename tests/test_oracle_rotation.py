"""Pins for the oracle's randomised Walsh-Hadamard rotation."""
import numpy as np
import pytest
import scipy.linalg

from oracle import rotation, rng


@pytest.mark.parametrize("d", [1, 2, 4, 8, 64, 128, 256, 512])
def test_matches_scipy_sylvester_hadamard(d):
    assert np.array_equal(rotation.hadamard(d), scipy.linalg.hadamard(d).astype(float))


@pytest.mark.parametrize("d", [2, 16, 64])
def test_entries_brute_force_popcount(d):
    h = rotation.hadamard(d)
    for i in range(d):
        for j in range(d):
            assert h[i, j] == (-1) ** bin(i & j).count("1")


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_h_squared_is_d_identity(d):
    h = rotation.hadamard(d)
    assert np.array_equal(h @ h, d * np.eye(d))


@pytest.mark.parametrize("d", [64, 128, 512])
def test_rotation_orthogonal_and_inverse(d):
    g = np.random.default_rng(d)
    x = g.standard_normal((50, d)) * g.lognormal(size=(50, 1))
    s = rng.signs(3, d)
    y = rotation.rotate(x, s)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12, atol=0)
    assert np.allclose(rotation.unrotate(y, s), x, rtol=0, atol=1e-12)
    # plain normalised WHT is an involution
    ones = np.ones(d)
    assert np.allclose(rotation.rotate(rotation.rotate(x, ones), ones), x, atol=1e-12)


@pytest.mark.parametrize("d", [64, 128])
def test_first_basis_vector_maps_to_constant(d):
    e0 = np.zeros(d)
    e0[0] = 1.0
    assert np.allclose(rotation.rotate(e0, np.ones(d)) * np.sqrt(d), np.ones(d), atol=0)


def test_signs_applied_before_transform():
    d = 32
    s = rng.signs(9, d)
    x = np.random.default_rng(1).standard_normal(d)
    h = scipy.linalg.hadamard(d).astype(float)
    assert np.allclose(rotation.rotate(x, s), h @ (s * x) / np.sqrt(d), atol=1e-13)
    assert np.allclose(rotation.unrotate(x, s), s * (h @ x) / np.sqrt(d), atol=1e-13)
