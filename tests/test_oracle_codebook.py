"""Pins for the oracle's Lloyd-Max codebook over the rotated-coordinate density."""
import numpy as np
import pytest
from scipy import integrate, special, stats

from oracle import codebook
from conftest import golden


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_density_normalised_and_cdf_consistent(d):
    tot, _ = integrate.quad(codebook.pdf, -1, 1, args=(d,), points=[0.0], epsabs=1e-13)
    assert abs(tot - 1.0) < 1e-10
    for x in [-0.3, -0.05, 0.0, 0.02, 0.2]:
        val, _ = integrate.quad(codebook.pdf, -1, x, args=(d,), epsabs=1e-13)
        assert abs(codebook.cdf(x, d) - val) < 1e-10


@pytest.mark.parametrize("d", [64, 128])
def test_density_matches_random_unit_vectors(d):
    """The coordinate of a uniformly random unit vector follows f_d (KS test)."""
    g = np.random.default_rng(0)
    x = g.standard_normal((200_000, d))
    coord = x[:, 0] / np.linalg.norm(x, axis=1)
    res = stats.kstest(coord, lambda t: codebook.cdf(t, d))
    assert res.pvalue > 1e-3


@pytest.mark.parametrize("d", [16, 64, 128, 512])
def test_density_moments_of_uniform_sphere(d):
    """E[x^2] = 1/d and E[x^4] = 3/(d(d+2)) for a coordinate of a uniform unit vector."""
    m2, _ = integrate.quad(lambda x: x * x * codebook.pdf(x, d), -1, 1, epsabs=1e-15)
    m4, _ = integrate.quad(lambda x: x ** 4 * codebook.pdf(x, d), -1, 1, epsabs=1e-15)
    assert abs(m2 * d - 1.0) < 1e-9
    assert abs(m4 * d * (d + 2) / 3.0 - 1.0) < 1e-9


@pytest.mark.parametrize("d", [32, 64, 128, 256, 512])
def test_one_bit_closed_form(d):
    c, b = codebook.lloyd_max(d, 1)
    exact = np.exp(special.gammaln(d / 2) - special.gammaln((d + 1) / 2)) / np.sqrt(np.pi)
    assert np.allclose(c, [-exact, exact], rtol=1e-12, atol=0)
    assert b.shape == (1,) and b[0] == 0.0


@pytest.mark.parametrize("d,bits", [(64, 2), (128, 2), (128, 3), (256, 2), (512, 3), (128, 4), (64, 4), (512, 4),
                                    (64, 5), (128, 6), (512, 7), (128, 8)])
def test_fixed_point_conditions_by_quadrature(d, bits):
    c, b = codebook.lloyd_max(d, bits)
    k = 1 << bits
    assert c.shape == (k,) and b.shape == (k - 1,)
    assert np.all(np.diff(c) > 0)
    assert np.array_equal(c, -c[::-1])
    assert np.allclose(b, 0.5 * (c[:-1] + c[1:]), atol=0)
    edges = np.concatenate(([-1.0], b, [1.0]))
    for j in range(k):
        num, _ = integrate.quad(lambda x: x * codebook.pdf(x, d), edges[j], edges[j + 1], epsabs=1e-15, epsrel=1e-13)
        den, _ = integrate.quad(lambda x: codebook.pdf(x, d), edges[j], edges[j + 1], epsabs=1e-15, epsrel=1e-13)
        assert abs(num / den - c[j]) < 1e-9 * np.sqrt(1.0 / d) + 1e-12


def test_gaussian_limit_matches_max_1960():
    """sqrt(d) * c_d tends to the Gaussian Lloyd-Max levels of Max (1960)."""
    table = golden("gaussian_lloyd_max.json")
    d = 1 << 14
    for k_str, pos in table["levels"].items():
        bits = int(k_str).bit_length() - 1
        c, _ = codebook.lloyd_max(d, bits)
        got = np.sqrt(d) * c[len(c) // 2:]
        assert np.allclose(got, pos, atol=2e-3), (k_str, got, pos)


def test_codebook_is_mse_optimal_among_perturbations():
    d = 128
    c, b = codebook.lloyd_max(d, 2)
    g = np.random.default_rng(5)
    x = g.standard_normal((400_000, d))
    coord = (x[:, 0] / np.linalg.norm(x, axis=1))

    def mse(cc):
        bb = 0.5 * (cc[:-1] + cc[1:])
        return np.mean((coord - cc[np.searchsorted(bb, coord)]) ** 2)

    base = mse(c)
    for eps in [0.05, -0.05]:
        assert mse(c * (1 + eps)) > base


@pytest.mark.parametrize("bits", [1, 2, 3])
def test_symmetric_codebook_is_odd_parity_combination(bits):
    # A codebook with c[K-1-i] = -c[i] is odd under flipping every index bit, so in the +-1
    # variables P_i = 1 - 2 b_i it is a combination of odd parity products only: one plane per
    # bit for 1 and 2 bits, the three planes plus P0 P1 P2 for 3 bits (Walsh expansion).
    import itertools
    c, _ = codebook.lloyd_max(128, bits)
    K = 1 << bits
    idx = np.arange(K)
    P = [1 - 2 * ((idx >> i) & 1) for i in range(bits)]  # P[i] for bit i (bit 0 = lowest)
    for r in range(bits + 1):
        for S in itertools.combinations(range(bits), r):
            chi = np.prod([P[i] for i in S], axis=0) if S else np.ones(K)
            coef = float(np.dot(c, chi)) / K
            if r % 2 == 0:
                assert abs(coef) < 1e-12, (S, coef)
    recon = np.zeros(K)
    for r in range(1, bits + 1, 2):
        for S in itertools.combinations(range(bits), r):
            chi = np.prod([P[i] for i in S], axis=0)
            recon += float(np.dot(c, chi)) / K * chi
    assert np.allclose(recon, c, atol=1e-12)


@pytest.mark.parametrize("d", [64, 512])
def test_large_codebooks_approach_the_panter_dite_limit(d):
    """High-resolution theory (Panter & Dite 1951): the optimal K-level quantiser's MSE tends to
    (1/12) (int f^(1/3))^3 / K^2.  The 32..256-level codebooks approach it from below, the gap
    roughly halving per bit."""
    pdc, _ = integrate.quad(lambda x: codebook.pdf(x, d) ** (1 / 3), -1, 1, points=[0.0], limit=200)
    limit = pdc ** 3 / 12
    ratios = []
    for bits in (5, 6, 7, 8):
        c, b = codebook.lloyd_max(d, bits)
        edges = np.concatenate(([-1.0], b, [1.0]))
        mse = sum(integrate.quad(lambda x: (x - c[j]) ** 2 * codebook.pdf(x, d), edges[j], edges[j + 1],
                                 epsabs=1e-18)[0] for j in range(len(c)))
        ratios.append(mse * 4 ** bits / limit)
    assert all(0.9 < r < 1.0 for r in ratios) and ratios[-1] > 0.99
    gaps = [1 - r for r in ratios]
    assert all(0.4 < gaps[i + 1] / gaps[i] < 0.6 for i in range(3))


@pytest.mark.parametrize("d,bits", [(64, 5), (512, 8)])
def test_large_codebook_is_a_fixed_point_of_lloyds_map(d, bits):
    """Lloyd's map (midpoint boundaries, then conditional means) leaves the solved codebook where it
    is: 1000 iterations from it move no centroid by more than 1e-10 / sqrt(d).  (The drift that
    remains is rounding in the far-tail cell probabilities, which Lloyd's slow contraction at 256
    levels does not damp; a wrong fixed point moves by orders of magnitude more.)"""
    c0, _ = codebook.lloyd_max(d, bits)
    c = c0.copy()
    for _ in range(1000):
        edges = np.concatenate(([-1.0], 0.5 * (c[:-1] + c[1:]), [1.0]))
        p = codebook.cdf(edges[1:], d) - codebook.cdf(edges[:-1], d)
        c = codebook.partial_first_moment(edges[:-1], edges[1:], d) / p
    assert np.max(np.abs(c - c0)) * np.sqrt(d) < 1e-10

