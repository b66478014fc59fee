"""Paged compressed KV cache: encoding whole token ranges into a pool (oracle).

The write path compresses tokens in page-aligned batches (the pages flush
128 tokens at a time, "turboquant-bench" technical details: batch flush of
128 tokens; turboquant vLLM guide, §5.1: decode tokens collect in a ring
buffer of ``buffer_size = 128``).  Here any page-aligned range may be
encoded; the ring semantics live in ``ring_split``.
"""
from __future__ import annotations

import numpy as np

from . import layout, quant

RING = 128


def ring_split(length: int, ring: int = RING):
    """(n_compressed, n_buffered) for a sequence of ``length`` tokens.

    Reading of "keep the newest 128 tokens exact" + "flush 128 at a time":
    a full ring is flushed only when a new token arrives, so the buffer
    always holds between 1 and 128 tokens once the sequence is non-empty.
    """
    if length <= 0:
        return 0, 0
    n_c = ring * ((length - 1) // ring)
    return n_c, length - n_c


def encode_main_range(pool, block_table, start, k16, v16, signs, centroids, s_mat, group=32):
    """Encode fp16 k/v [B, Hkv, T, d] for positions start .. start+T-1 into ``pool``.

    ``pool`` is uint8 [num_blocks, Hkv, tile]; ``start`` and T are multiples
    of 16.  Returns the key-encoder dict (for boundary diagnostics).
    """
    k16 = np.asarray(k16, dtype=np.float16)
    bsz, hkv, t, d = k16.shape
    assert start % layout.P == 0 and t % layout.P == 0
    enc = quant.encode_keys(k16, signs, centroids, s_mat)
    vq, vs, vmn = quant.encode_values(v16, group)
    npg = t // layout.P
    tiles = layout.pack_main_tiles(
        enc["idx"].reshape(bsz, hkv, npg, 16, d),
        enc["sigma"].reshape(bsz, hkv, npg, 16, d),
        vq.reshape(bsz, hkv, npg, 16, d),
        vs.reshape(bsz, hkv, npg, 16, d // group),
        vmn.reshape(bsz, hkv, npg, 16, d // group),
        enc["n_k"].reshape(bsz, hkv, npg, 16),
        enc["n_r"].reshape(bsz, hkv, npg, 16),
    )
    pages = start // layout.P + np.arange(npg)
    blocks = np.asarray(block_table)[:, pages]  # [B, npg]
    pool[blocks[:, None, :], np.arange(hkv)[None, :, None]] = tiles
    return enc


def encode_alt_range(pool, block_table, start, k16, v16, signs, centroids3):
    """Alternate layout: encode fp16 k/v [B, Hkv, T, d] into ``pool``."""
    k16 = np.asarray(k16, dtype=np.float16)
    bsz, hkv, t, d = k16.shape
    assert start % layout.P == 0 and t % layout.P == 0
    kq, ks, kmn = quant.encode_alt_keys(k16)
    venc = quant.encode_alt_values(v16, signs, centroids3)
    npg = t // layout.P
    tiles = layout.pack_alt_tiles(
        kq.reshape(bsz, hkv, npg, 16, d),
        ks.reshape(bsz, hkv, npg, 16, d // 32),
        kmn.reshape(bsz, hkv, npg, 16, d // 32),
        venc["idx"].reshape(bsz, hkv, npg, 16, d),
        venc["n_v"].reshape(bsz, hkv, npg, 16),
    )
    pages = start // layout.P + np.arange(npg)
    blocks = np.asarray(block_table)[:, pages]
    pool[blocks[:, None, :], np.arange(hkv)[None, :, None]] = tiles
    return venc


def read_main(pool, block_table, b, n_c, d):
    """Unpack the first n_c tokens of sequence b: fields [Hkv, n_c, ...]."""
    npg = n_c // layout.P
    tiles = pool[np.asarray(block_table)[b, :npg]]  # [npg, Hkv, tile]
    f = layout.unpack_main_tiles(tiles, d)
    out = {}
    for key, val in f.items():
        val = np.moveaxis(val, 1, 0)  # [Hkv, npg, 16, ...]
        out[key] = val.reshape((val.shape[0], npg * layout.P) + val.shape[3:])
    return out


def read_alt(pool, block_table, b, n_c, d):
    npg = n_c // layout.P
    tiles = pool[np.asarray(block_table)[b, :npg]]
    f = layout.unpack_alt_tiles(tiles, d)
    out = {}
    for key, val in f.items():
        val = np.moveaxis(val, 1, 0)
        out[key] = val.reshape((val.shape[0], npg * layout.P) + val.shape[3:])
    return out
