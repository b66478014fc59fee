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
    kbits, vbits = layout.main_bits(pool.shape[-1], d, key_bits_of(centroids))
    enc = quant.encode_keys(k16, signs, centroids, s_mat)
    vq, vs, vmn = quant.encode_values(v16, group, vbits)
    npg = t // layout.P
    tiles = layout.pack_main_tiles(
        enc["idx"].reshape(bsz, hkv, npg, 16, d),
        enc["sigma"].reshape(bsz, hkv, npg, 16, d),
        vq.reshape(bsz, hkv, npg, 16, d),
        vs.reshape(bsz, hkv, npg, 16, d // group),
        vmn.reshape(bsz, hkv, npg, 16, d // group),
        enc["n_k"].reshape(bsz, hkv, npg, 16),
        enc["n_r"].reshape(bsz, hkv, npg, 16),
        vbits,
        kbits,
    )
    pages = start // layout.P + np.arange(npg)
    blocks = np.asarray(block_table)[:, pages]  # [B, npg]
    pool[blocks[:, None, :], np.arange(hkv)[None, :, None]] = tiles
    return enc


def value_bits_of(centroids) -> int:
    """Alternate-layout value bits for a Lloyd-Max codebook of 2^bits centroids (2 to 8 bits: the
    vllm-metal TurboQuant guide's q2_0 .. q8_0 value formats)."""
    k = len(centroids)
    assert k in (4, 8, 16, 32, 64, 128, 256), k
    return k.bit_length() - 1


def encode_alt_range(pool, block_table, start, k16, v16, signs, centroids3, key_signed=False):
    """Alternate layout: encode fp16 k/v [B, Hkv, T, d] into ``pool`` (value bits from the codebook
    size: 4 to 256 centroids; key bits from the pool's tile size: 8, 5, 4, 2, or 16 for fp16
    keys; key_signed: 2-bit keys as int2 instead of uint2)."""
    k16 = np.asarray(k16, dtype=np.float16)
    bsz, hkv, t, d = k16.shape
    assert start % layout.P == 0 and t % layout.P == 0
    vb = value_bits_of(centroids3)
    kb = layout.alt_key_bits(pool.shape[-1], d, vb)
    kq, ks, kmn = quant.encode_alt_keys(k16, bits=kb, signed=key_signed)
    venc = quant.encode_alt_values(v16, signs, centroids3)
    npg = t // layout.P
    tiles = layout.pack_alt_tiles(
        kq.reshape(bsz, hkv, npg, 16, d),
        None if ks is None else ks.reshape(bsz, hkv, npg, 16, d // 32),
        None if kmn is None else kmn.reshape(bsz, hkv, npg, 16, d // 32),
        venc["idx"].reshape(bsz, hkv, npg, 16, d),
        venc["n_v"].reshape(bsz, hkv, npg, 16),
        vb,
        kb,
    )
    pages = start // layout.P + np.arange(npg)
    blocks = np.asarray(block_table)[:, pages]
    pool[blocks[:, None, :], np.arange(hkv)[None, :, None]] = tiles
    return venc


def key_bits_of(centroids) -> int:
    """Main-layout key bits for a Lloyd-Max codebook: its index bits plus the QJL bit."""
    k = len(centroids)
    assert k in (2, 4, 8), k
    return k.bit_length()


def read_main(pool, block_table, b, n_c, d, kbits=None):
    """Unpack the first n_c tokens of sequence b: fields [Hkv, n_c, ...]."""
    npg = n_c // layout.P
    tiles = pool[np.asarray(block_table)[b, :npg]]  # [npg, Hkv, tile]
    f = layout.unpack_main_tiles(tiles, d, kbits)
    out = {}
    for key, val in f.items():
        val = np.moveaxis(val, 1, 0)  # [Hkv, npg, 16, ...]
        out[key] = val.reshape((val.shape[0], npg * layout.P) + val.shape[3:])
    return out


def read_alt(pool, block_table, b, n_c, d, vbits=None):
    npg = n_c // layout.P
    tiles = pool[np.asarray(block_table)[b, :npg]]
    f = layout.unpack_alt_tiles(tiles, d, vbits)
    out = {}
    for key, val in f.items():
        val = np.moveaxis(val, 1, 0)
        out[key] = val.reshape((val.shape[0], npg * layout.P) + val.shape[3:])
    return out


def materialize_main(pool, block_table, b, n_c, ring_k, ring_v, n_buf, signs, centroids, s_mat, d):
    """Dense history of sequence b as float64 (k, v) [Hkv, n_c + n_buf, d] (main layout).

    Prefill materialisation (vllm-metal TurboQuant guide, advanced settings): the
    compressed tokens become the explicit reconstruction k^ (quant.dequant_keys) and
    mn + s q (quant.group_dequant); the ring tokens follow unchanged.
    """
    f = read_main(pool, block_table, b, n_c, d, key_bits_of(centroids)) if n_c else None
    hkv = pool.shape[1]
    ks, vs = [], []
    for g in range(hkv):
        kk, vv = [], []
        if n_c:
            enc = {"idx": f["idx"][g], "sigma": f["sigma"][g], "n_k": f["n_k"][g], "n_r": f["n_r"][g]}
            kk.append(quant.dequant_keys(enc, signs, centroids, s_mat))
            vv.append(quant.group_dequant(f["vq"][g], f["vs"][g], f["vmn"][g], 32))
        if n_buf:
            kk.append(np.asarray(ring_k[b, g, :n_buf], np.float64))
            vv.append(np.asarray(ring_v[b, g, :n_buf], np.float64))
        ks.append(np.concatenate(kk, axis=0) if kk else np.zeros((0, d)))
        vs.append(np.concatenate(vv, axis=0) if vv else np.zeros((0, d)))
    return np.stack(ks), np.stack(vs)


def materialize_alt(pool, block_table, b, n_c, ring_k, ring_v, n_buf, signs, centroids3, d):
    """Dense history of sequence b as float64 (k, v) [Hkv, n_c + n_buf, d] (alternate layout)."""
    f = read_alt(pool, block_table, b, n_c, d, value_bits_of(centroids3)) if n_c else None
    hkv = pool.shape[1]
    ks, vs = [], []
    for g in range(hkv):
        kk, vv = [], []
        if n_c:
            kk.append(quant.alt_keys({key: val[g] for key, val in f.items()}))
            vv.append(quant.dequant_alt_values(f["vidx"][g], f["n_v"][g], signs, centroids3))
        if n_buf:
            kk.append(np.asarray(ring_k[b, g, :n_buf], np.float64))
            vv.append(np.asarray(ring_v[b, g, :n_buf], np.float64))
        ks.append(np.concatenate(kk, axis=0) if kk else np.zeros((0, d)))
        vs.append(np.concatenate(vv, axis=0) if vv else np.zeros((0, d)))
    return np.stack(ks), np.stack(vs)
