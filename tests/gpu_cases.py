"""Scenario builders and comparison helpers for the GPU parity tests.

Inputs come from ``synth``; expected values from ``oracle``; nothing here
computes the method.  Bit extraction for comparisons is written out here so
that CUDA output is never fed through oracle code.
"""
import numpy as np
import torch

import synth
from oracle import cache, codebook, layout, quant, rng

MARGIN = 1e-5  # oracle values this close to a decision boundary may legitimately differ


def oracle_tables(seed, d, layout_main=True, key_bits=3, value_bits=3):
    bits = key_bits - 1 if layout_main else value_bits
    c, _ = codebook.lloyd_max(d, bits)
    c32 = c.astype(np.float32)
    signs = rng.signs(seed, d).astype(np.float32)
    sketch = rng.gaussian_matrix(seed, d, d) if layout_main else None
    return c32, signs, sketch


def make_ctx(tq, layout_main, d, hq, hkv, seed, value_bits=None, key_bits=None):
    c32, signs, sketch = oracle_tables(seed, d, layout_main, key_bits or 3, value_bits or 3)
    lay = tq.TQ_LAYOUT_MAIN if layout_main else tq.TQ_LAYOUT_ALT
    ctx = tq.Context(lay, d, hq, hkv, seed, centroids=c32, signs=signs, sketch=sketch, value_bits=value_bits,
                     key_bits=key_bits)
    return ctx, c32.astype(np.float64), signs.astype(np.float64), sketch


def to_dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


# ---------------------------------------------------------------- bit helpers (test-local)
def plane_bits(words_u32):
    """uint32 [..., n/32] -> bits [..., n] with coordinate 32w+2j+e at bit 16e+j."""
    w = words_u32.astype(np.uint64)[..., None, None]
    sh = (16 * np.arange(2)[None, :] + np.arange(16)[:, None]).astype(np.uint64)
    b = (w >> sh) & np.uint64(1)
    return b.reshape(words_u32.shape[:-1] + (words_u32.shape[-1] * 32,)).astype(np.uint8)


def main_fields(tiles, d, kb=None):
    """Fields of main-layout tiles; kb = key bits (2, 3 or 4), taken from the tile size when not
    given (the size alone cannot tell 4-bit keys with 2-bit values from 2-bit keys with 4-bit
    values)."""
    t = np.ascontiguousarray(tiles)
    lead = t.shape[:-1]
    o_n = t.shape[-1] - 64  # norms sit in the last 64 bytes (2- or 4-bit value codes before them)
    if kb is None:  # (2 kb + 2 vb + 2) d + 64 with kb in {2, 3}, vb in {2, 4}
        units = (t.shape[-1] - 64) // (2 * d) - 1  # kb + vb
        kb = 3 if units in (5, 7) else 2
    w = lambda off, n: np.ascontiguousarray(t[..., off:off + n]).view("<u4")
    pl = [plane_bits(w(2 * d * i, 2 * d).reshape(lead + (16, d // 32))) for i in range(kb)]
    idx = np.zeros_like(pl[0])
    for i in range(kb - 1):
        idx = 2 * idx + pl[i]
    return {
        "idx": idx,
        "sigma": pl[kb - 1],
        "v_bytes": t[..., 2 * kb * d:o_n],
        "kn": np.ascontiguousarray(t[..., o_n:o_n + 32]).view("<i2"),
        "rn": np.ascontiguousarray(t[..., o_n + 32:o_n + 64]).view("<i2"),
    }


def alt_fields(tiles, d, kb=8):
    """Fields of alternate-layout tiles with kb-bit keys, or fp16 keys for kb = 16 (value bits vb
    from the size: key bytes + 2 vb d + 32)."""
    t = np.ascontiguousarray(tiles)
    lead = t.shape[:-1]
    o_vi = 32 * d if kb == 16 else (2 * kb + 2) * d
    vb = (t.shape[-1] - o_vi - 32) // (2 * d)
    o_n = o_vi + 2 * vb * d
    vi = t[..., o_vi:o_n].reshape(lead + (16, vb * d // 8))
    bits = np.unpackbits(vi, axis=-1, bitorder="little").reshape(lead + (16, d, vb)).astype(np.uint8)
    idx = sum(bits[..., i].astype(np.int32) << i for i in range(vb)).astype(np.uint8)
    return {
        "k_bytes": t[..., :o_vi],  # key codes and their (scale, minimum) pairs, or fp16 keys
        "vidx": idx,
        "vn": np.ascontiguousarray(t[..., o_n:o_n + 32]).view("<i2"),
    }


def near_boundary(y, centroids):
    b = 0.5 * (centroids[:-1] + centroids[1:])
    return np.min(np.abs(y[..., None] - b), axis=-1) < MARGIN


def tile_index(bt, starts, n_tok):
    """(block ids [B, pages]) of the pages holding tokens start..start+n_tok-1 of each sequence."""
    pages = np.arange(n_tok // 16)
    return np.stack([bt[b, starts[b] // 16 + pages] for b in range(len(starts))])


def allclose_report(got, ref, atol=2e-3, rtol=1e-3):
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    return (not bad.any()), float(err.max()) if err.size else 0.0, int(bad.sum())


# ---------------------------------------------------------------- decode scenarios
def build_main_cache(seed, d, hkv, lengths, centroids, signs, sketch, shuffled=True, extra_blocks=0, value_bits=2,
                     key_bits=3, v_scale=1.0):
    """Oracle-encoded pool + ring for sequences of the given total lengths (values multiplied by
    v_scale before rounding to fp16, for large-magnitude value groups)."""
    bsz = len(lengths)
    lmax = max(max(lengths), 1)
    t_all = ((lmax + 15) // 16) * 16
    k, v = synth.kv_main(seed, bsz, hkv, t_all, d)
    if v_scale != 1.0:
        v = (v.astype(np.float32) * np.float32(v_scale)).astype(np.float16)
    max_blocks = max(t_all // 16, 1)
    bt = synth.block_table(seed, bsz, max_blocks, shuffled)
    nblk = bsz * max_blocks + extra_blocks
    pool = np.zeros((nblk, hkv, layout.main_tile_bytes(d, value_bits, key_bits)), np.uint8)
    n_c = np.zeros(bsz, np.int32)
    n_b = np.zeros(bsz, np.int32)
    ring_k = np.zeros((bsz, hkv, 128, d), np.float16)
    ring_v = np.zeros_like(ring_k)
    for b, L in enumerate(lengths):
        nc, nb = cache.ring_split(L)
        n_c[b], n_b[b] = nc, nb
        if nc:
            cache.encode_main_range(pool, bt[b:b + 1], 0, k[b:b + 1, :, :nc], v[b:b + 1, :, :nc], signs, centroids, sketch)
        ring_k[b, :, :nb] = k[b, :, nc:nc + nb]
        ring_v[b, :, :nb] = v[b, :, nc:nc + nb]
    return dict(k=k, v=v, bt=bt, pool=pool, n_c=n_c, n_b=n_b, ring_k=ring_k, ring_v=ring_v, max_ctx=int(n_c.max()) if bsz else 0)


def build_alt_cache(seed, d, hkv, lengths, centroids3, signs, shuffled=True, key_bits=8, key_signed=False):
    bsz = len(lengths)
    t_all = ((max(lengths) + 15) // 16) * 16
    k, v = synth.kv_alt(seed, bsz, hkv, t_all, d)
    max_blocks = t_all // 16
    bt = synth.block_table(seed, bsz, max_blocks, shuffled)
    pool = np.zeros((bsz * max_blocks, hkv, layout.alt_tile_bytes(d, cache.value_bits_of(centroids3), key_bits)),
                    np.uint8)
    n_c = np.array(lengths, np.int32)
    for b, L in enumerate(lengths):
        cache.encode_alt_range(pool, bt[b:b + 1], 0, k[b:b + 1, :, :L], v[b:b + 1, :, :L], signs, centroids3,
                               key_signed=key_signed)
    return dict(k=k, v=v, bt=bt, pool=pool, n_c=n_c, max_ctx=int(n_c.max()))
