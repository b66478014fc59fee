"""Seeded synthetic inputs for the TurboQuant-style KV-cache workloads.

This module holds no arithmetic of the method: it draws raw keys, values,
queries, context lengths and block tables and nothing else.  The oracle
tests, the CUDA parity tests and the benchmark all take their inputs from
here, so both sides see identical fp16 arrays.

Recipe (the workloads' shapes are those of the Qwen2.5/Qwen3 decode
geometries named by the benchmark configurations):

* keys / values (main layout): iid N(0, 1); per KV head, 4 outlier channels
  (the first 4 entries of a seeded permutation of ``head_dim``, drawn
  separately for K and for V) are multiplied by 10; every (token, KV head)
  vector is then multiplied by one log-normal factor exp(N(0, 0.5^2));
  finally rounded to fp16 (round-to-nearest-even).
* keys / values (alternate layout): iid N(0, 1) where each entry is, with
  probability 0.02, replaced by a Student-t draw with 3 degrees of freedom;
  rounded to fp16.
* queries: iid N(0, 1) rounded to fp16.
* ragged context lengths: uniform integers in [lo, hi] (inclusive).
* block tables: identity, or a seeded random permutation of the physical
  blocks (each sequence gets ``max_blocks`` distinct physical blocks).

Every generator takes an integer seed plus integer "stream" words and builds
its numpy ``Generator`` from ``SeedSequence([seed, *streams])`` so that
different tensors of one workload never share random numbers.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng_for",
    "kv_main",
    "kv_alt",
    "queries",
    "ragged_lengths",
    "block_table",
    "random_codes",
]

# stream tags (arbitrary distinct integers)
_K, _V, _Q, _LEN, _BT, _CODES = 11, 12, 13, 14, 15, 16


def rng_for(seed: int, *streams: int) -> np.random.Generator:
    """numpy Generator for (seed, streams...)."""
    return np.random.default_rng(np.random.SeedSequence([int(seed)] + [int(s) for s in streams]))


def _outlier_lognormal(rng: np.random.Generator, batch: int, n_kv: int, n_tok: int, d: int) -> np.ndarray:
    x = rng.standard_normal((batch, n_kv, n_tok, d), dtype=np.float32)
    for h in range(n_kv):
        ch = rng.permutation(d)[:4]
        x[:, h, :, ch] *= np.float32(10.0)
    scale = np.exp(rng.normal(0.0, 0.5, size=(batch, n_kv, n_tok, 1))).astype(np.float32)
    x *= scale
    return x.astype(np.float16)


def kv_main(seed: int, batch: int, n_kv: int, n_tok: int, d: int, layer: int = 0):
    """(k, v) fp16 arrays [batch, n_kv, n_tok, d] with outlier channels and log-normal norms."""
    k = _outlier_lognormal(rng_for(seed, layer, _K), batch, n_kv, n_tok, d)
    v = _outlier_lognormal(rng_for(seed, layer, _V), batch, n_kv, n_tok, d)
    return k, v


def _student_mix(rng: np.random.Generator, shape, frac: float = 0.02) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    mask = rng.random(shape, dtype=np.float32) < np.float32(frac)
    n = int(mask.sum())
    if n:
        x[mask] = rng.standard_t(3.0, size=n).astype(np.float32)
    return x.astype(np.float16)


def kv_alt(seed: int, batch: int, n_kv: int, n_tok: int, d: int, layer: int = 0):
    """(k, v) fp16 arrays [batch, n_kv, n_tok, d]: N(0,1) with 2% Student-t(3) entries."""
    shape = (batch, n_kv, n_tok, d)
    k = _student_mix(rng_for(seed, layer, _K), shape)
    v = _student_mix(rng_for(seed, layer, _V), shape)
    return k, v


def queries(seed: int, batch: int, n_q: int, d: int, layer: int = 0, step: int = 0) -> np.ndarray:
    """fp16 queries [batch, n_q, d], iid N(0, 1)."""
    rng = rng_for(seed, layer, _Q, step)
    return rng.standard_normal((batch, n_q, d), dtype=np.float32).astype(np.float16)


def ragged_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """int64 lengths, uniform on [lo, hi] inclusive."""
    return rng_for(seed, _LEN).integers(lo, hi, size=batch, endpoint=True)


def block_table(seed: int, batch: int, max_blocks: int, shuffled: bool) -> np.ndarray:
    """int32 [batch, max_blocks] physical block ids; a permutation of range(batch * max_blocks)."""
    n = batch * max_blocks
    ids = np.arange(n, dtype=np.int32)
    if shuffled:
        ids = rng_for(seed, _BT).permutation(n).astype(np.int32)
    return ids.reshape(batch, max_blocks)


def random_codes(seed: int, n: int, bits: int) -> np.ndarray:
    """uint8 array of n uniform codes in [0, 2**bits)."""
    return rng_for(seed, _CODES, bits).integers(0, 1 << bits, size=n, dtype=np.uint8)
