"""Randomised Walsh-Hadamard rotation (oracle, float64).

The pages rotate every vector by a random orthogonal transform before scalar
quantisation so that its coordinates look alike ("TurboQuant-MLX overview",
PolarQuant step 1: randomised Hadamard rotation; turboquant vLLM guide, §二
step 1: random orthogonal rotation).  The plain reading used here:

    y = H_d (D * x) / sqrt(d)

with D a diagonal of random signs and H_d the Sylvester-ordered Hadamard
matrix, H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]], i.e.
H[i, j] = (-1) ** popcount(i & j).  Because H_d is symmetric and
H_d H_d = d I, the inverse is x = D * (H_d y) / sqrt(d).

The matrix is built explicitly; no fast transform is used here.
"""
from __future__ import annotations

import numpy as np


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (a power of two), float64."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """y = H (D x) / sqrt(d) along the last axis."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = hadamard(d)
    return ((x * np.asarray(signs, dtype=np.float64)) @ h.T) / np.sqrt(d)


def unrotate(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """x = D (H y) / sqrt(d) along the last axis (inverse of ``rotate``)."""
    y = np.asarray(y, dtype=np.float64)
    d = y.shape[-1]
    h = hadamard(d)
    return (y @ h.T) / np.sqrt(d) * np.asarray(signs, dtype=np.float64)
