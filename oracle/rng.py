"""Counter-based generator for the method's random tables (oracle).

The method draws one random-sign diagonal D (length d) and one Gaussian
sketch matrix S (m x d, iid N(0, 1)) per layer (turboquant vLLM guide, §八:
"random orthogonal rotation + QJL matrix"; §二 step 3, QJL residual sign
bits).  The pages fix no generator, so both sides of this project implement
the same published one:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; S. Vigna's reference C code splitmix64.c):
  state += 0x9E3779B97F4A7C15; z = state;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
  output z ^ (z >> 31).
  Output n (n = 0, 1, ...) of a generator with initial state s0 is therefore
  mix(s0 + (n + 1) * gamma), which is what ``words`` evaluates directly.
* Box-Muller (Box & Muller, 1958) for normal deviates.

Table recipe (this project's definition):

* stream word n of (seed, stream) = SplitMix64 output n for the initial state
  s0 = (seed + stream * 2**40) mod 2**64;
* D_i = -1 if bit 63 of word i of stream 1 is set, else +1   (i < d);
* for pair k, a = word 2k and b = word 2k+1 of stream 2,
  u1 = ((a >> 11) + 1) * 2**-53, u2 = (b >> 11) * 2**-53,
  R = sqrt(-2 ln u1), S_flat[2k] = R cos(2 pi u2), S_flat[2k+1] = R sin(2 pi u2);
  S = S_flat reshaped to (m, d) row-major, then rounded to float32.
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MASK = (1 << 64) - 1


def mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on uint64 arrays."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def words(seed: int, stream: int, n: int) -> np.ndarray:
    """First n SplitMix64 outputs for (seed, stream), uint64."""
    s0 = (int(seed) + int(stream) * (1 << 40)) & MASK
    idx = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(s0) + idx * np.uint64(GAMMA)
    return mix(state)


def signs(seed: int, d: int) -> np.ndarray:
    """Random-sign diagonal D as float64 +-1."""
    w = words(seed, 1, d)
    return np.where((w >> np.uint64(63)) != 0, -1.0, 1.0)


def gaussian_matrix(seed: int, m: int, d: int) -> np.ndarray:
    """S (m x d) iid N(0,1) by Box-Muller, rounded to float32."""
    n = m * d
    npairs = (n + 1) // 2
    w = words(seed, 2, 2 * npairs)
    a = w[0::2]
    b = w[1::2]
    u1 = ((a >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (b >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * npairs)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:n].reshape(m, d).astype(np.float32)
