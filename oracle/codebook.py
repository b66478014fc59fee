"""Lloyd-Max codebook for one coordinate of a rotated unit vector (oracle).

The key path maps each rotated coordinate to the nearest centroid of an
MSE-optimal scalar codebook precomputed for the "Beta distribution" of the
rotated coordinates (turboquant vLLM guide, §二 step 2, codebooks per head
dimension and bit width; "TurboQuant-MLX overview", PolarQuant step 2, 8
centroids at 3 bits; vllm-metal TurboQuant guide, quantisation principle
table).

Reading taken: after a uniformly random rotation, one coordinate x of a unit
vector in R^d has the density

    f_d(x) = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) * (1 - x^2)^((d-3)/2),  |x| <= 1,

(x^2 ~ Beta(1/2, (d-1)/2), which is the Beta distribution the page names).
The codebook is the Lloyd-Max fixed point for f_d:

    boundaries   b_j = (c_{j-1} + c_j) / 2
    centroids    c_j = E[x | b_j <= x < b_{j+1}]

iterated from a Gaussian-quantile start until the centroids move less than
1e-15.  Cell probabilities come from the regularised incomplete beta
function, the partial first moment from its closed form

    int_a^b x f_d(x) dx = C / (d-1) * ((1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)).

Centroids are returned in ascending order, index 0 = most negative, and made
exactly antisymmetric (c_j = -c_{K-1-j}), as the density is even.

From 32 levels up (the 5- to 8-bit value formats of the vllm-metal TurboQuant
guide, quantisation table: q5_0 .. q8_0 values), Lloyd's iteration contracts
too slowly to reach that tolerance in reasonable time, so the same two
conditions are solved by Newton's method: F(c) = c - T(c) with T_j the
conditional mean of cell j.  T_j depends only on the cell's edges a_j, b_j,
with dT/db = f(b)(b - T)/P and dT/da = f(a)(T - a)/P (P the cell probability),
and each inner edge is the midpoint of its two centroids, so the Jacobian is
tridiagonal.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_banded
from scipy.special import betainc, gammaln, ndtri


def density_const(d: int) -> float:
    """C_d = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2))."""
    return float(np.exp(gammaln(d / 2.0) - 0.5 * np.log(np.pi) - gammaln((d - 1) / 2.0)))


def pdf(x, d: int):
    x = np.asarray(x, dtype=np.float64)
    return density_const(d) * np.clip(1.0 - x * x, 0.0, None) ** ((d - 3) / 2.0)


def cdf(x, d: int):
    """P(X <= x) for the rotated-coordinate density."""
    x = np.clip(np.asarray(x, dtype=np.float64), -1.0, 1.0)
    half = 0.5 * betainc(0.5, (d - 1) / 2.0, x * x)
    return 0.5 + np.sign(x) * half


def partial_first_moment(a, b, d: int):
    """int_a^b x f_d(x) dx."""
    a = np.clip(np.asarray(a, dtype=np.float64), -1.0, 1.0)
    b = np.clip(np.asarray(b, dtype=np.float64), -1.0, 1.0)
    e = (d - 1) / 2.0
    return density_const(d) / (d - 1) * ((1.0 - a * a) ** e - (1.0 - b * b) ** e)


def _cell_means(c, d: int):
    """(T, edges, P): conditional means, edges and probabilities of the cells of centroids c."""
    edges = np.concatenate(([-1.0], 0.5 * (c[:-1] + c[1:]), [1.0]))
    p = cdf(edges[1:], d) - cdf(edges[:-1], d)
    return partial_first_moment(edges[:-1], edges[1:], d) / p, edges, p


def _newton(c, d: int, tol: float, max_iter: int = 100):
    """Fixed point c = T(c) by Newton's method with a tridiagonal Jacobian (step halved while the
    residual does not shrink)."""
    k = len(c)
    t, edges, p = _cell_means(c, d)
    f = c - t
    for _ in range(max_iter):
        if np.max(np.abs(f)) < tol:
            break
        a, b = edges[:-1], edges[1:]
        dta = pdf(a, d) * (t - a) / p  # dT_j / d a_j   (a_0 = -1 is fixed: pdf(-1) = 0)
        dtb = pdf(b, d) * (b - t) / p  # dT_j / d b_j   (b_{K-1} = 1 is fixed)
        # rows of I - dT/dc: a_j = (c_{j-1} + c_j)/2, b_j = (c_j + c_{j+1})/2
        ab = np.zeros((3, k))
        ab[0, 1:] = -0.5 * dtb[:-1]            # super-diagonal: -dT_j/dc_{j+1}
        ab[1, :] = 1.0 - 0.5 * (dta + dtb)     # diagonal
        ab[2, :-1] = -0.5 * dta[1:]            # sub-diagonal: -dT_j/dc_{j-1}
        step = solve_banded((1, 1), ab, -f)
        lam = 1.0
        while True:
            cn = c + lam * step
            tn, en, pn = _cell_means(cn, d)
            fn = cn - tn
            if np.all(np.diff(cn) > 0) and np.max(np.abs(fn)) < np.max(np.abs(f)) or lam < 1e-6:
                break
            lam *= 0.5
        c, t, edges, p, f = cn, tn, en, pn, fn
    return c


def lloyd_max(d: int, bits: int, tol: float = 1e-15, max_iter: int = 1_000_000):
    """(centroids[K], boundaries[K-1]) for K = 2**bits levels, float64."""
    if d < 4:
        raise ValueError("head dimension too small")
    k = 1 << bits
    c = ndtri((np.arange(k) + 0.5) / k) / np.sqrt(d)
    if bits >= 5:
        c = _newton(c, d, tol)
        c = 0.5 * (c - c[::-1])
        return c, 0.5 * (c[:-1] + c[1:])
    for _ in range(max_iter):
        edges = np.concatenate(([-1.0], 0.5 * (c[:-1] + c[1:]), [1.0]))
        p = cdf(edges[1:], d) - cdf(edges[:-1], d)
        m = partial_first_moment(edges[:-1], edges[1:], d)
        c_new = m / p
        done = np.max(np.abs(c_new - c)) < tol
        c = c_new
        if done:
            break
    c = 0.5 * (c - c[::-1])
    return c, 0.5 * (c[:-1] + c[1:])
