"""Bit packing and the paged tile layouts (oracle).

Generic low-bit streams (turboquant vLLM guide, §二 step 5, "4 values per
byte" at 2 bits; "TurboQuant-MLX overview", PolarQuant step 3, 3-bit
indices): value i of an n-value b-bit stream occupies stream bits
[b*i, b*i + b), least significant bit first, and stream bit k is bit
(k mod 8) of byte k // 8.  So 2-bit values 0,1,2,3 give the byte 0xE4, and
32 three-bit values fill exactly 12 bytes.

Page tiles.  A page holds P = 16 consecutive tokens of one sequence; a
tile is one page of one KV head.  The pool is ``uint8[num_blocks][Hkv][tile]``
and token position p of sequence b lives in tile
``(block_table[b][p // 16], kv_head)`` at slot ``p % 16``.  All multi-byte
fields are little-endian.

Main layout tile (d = head_dim = m), 12 d + 64 bytes = 16 x (0.75 d + 4):

    offset   size   plane
    0        2d     KH  high bit of each 2-bit Lloyd-Max key index
    2d       2d     KL  low bit of each key index
    4d       2d     KS  QJL sign bits sigma_j = [(S r)_j >= 0]
    6d       4d     VQ  2-bit value codes, one uint32 per dimension
    10d      2d     VSM per token and 32-group: fp16 scale, fp16 minimum
    12d      32     KN  fp16 key norm per token
    12d+32   32     RN  fp16 residual norm per token

  KH, KL, KS are token-major: token t's row is d/8 bytes at t*d/8, read as
  uint32 words; coordinate 32w + 2j + e (j < 16, e in {0, 1}) is bit
  16e + j of word w (even coordinates in the low half-word, odd ones in
  the high half-word).
  VQ is dimension-major: word i holds dimension i for the 16 tokens; the
  code of token 2j + e is at bits 16e + 2j and 16e + 2j + 1.
  VSM: token t, group g at byte (t * d/32 + g) * 4: scale then minimum.

Alternate layout tile, 24 d + 32 bytes = 16 x (1.5 d + 2):

    offset   size   plane
    0        16d    KQ  8-bit affine key codes, token-major (dimension i at byte i)
    16d      2d     KSM per token and 32-block: fp16 scale, fp16 minimum
    18d      6d     VI  3-bit value indices, per token a 3d/8-byte generic stream
    24d      32     VN  fp16 value norm per token

  With fp16 keys (kbits 16: keys kept exact and only the values quantised,
  the V-only mode of the "TurboQuant-MLX overview") KQ is 32d bytes of fp16
  keys and there is no KSM plane: 16 x (2d + vbits d/8 + 2) bytes.
"""
from __future__ import annotations

import numpy as np

P = 16  # tokens per page


# ---------------------------------------------------------------- generic streams
def pack_bits(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes (< 2**bits) into a little-endian LSB-first byte stream."""
    codes = np.asarray(codes, dtype=np.uint8).ravel()
    if bits < 1 or bits > 8:
        raise ValueError("bits must be in 1..8")
    if codes.size and int(codes.max()) >= (1 << bits):
        raise ValueError("code out of range")
    bitmat = ((codes[:, None] >> np.arange(bits, dtype=np.uint8)) & 1).astype(np.uint8)
    stream = bitmat.ravel()
    return np.packbits(stream, bitorder="little")


def unpack_bits(buf: np.ndarray, n: int, bits: int) -> np.ndarray:
    stream = np.unpackbits(np.asarray(buf, dtype=np.uint8), bitorder="little")[: n * bits]
    bitmat = stream.reshape(n, bits).astype(np.uint16)
    return (bitmat << np.arange(bits, dtype=np.uint16)).sum(axis=1).astype(np.uint8)


def packed_size(n: int, bits: int) -> int:
    return (n * bits + 7) // 8


def pack_rows(codes: np.ndarray, bits: int) -> np.ndarray:
    """``pack_bits`` applied to every row of codes [..., n] (n*bits % 8 == 0)."""
    codes = np.asarray(codes, dtype=np.uint8)
    n = codes.shape[-1]
    bitmat = ((codes[..., None] >> np.arange(bits, dtype=np.uint8)) & 1).astype(np.uint8)
    stream = bitmat.reshape(codes.shape[:-1] + (n * bits,))
    return np.packbits(stream, axis=-1, bitorder="little")


def unpack_rows(buf: np.ndarray, n: int, bits: int) -> np.ndarray:
    """Inverse of ``pack_rows``: bytes [..., n*bits/8] -> codes [..., n]."""
    buf = np.asarray(buf, dtype=np.uint8)
    stream = np.unpackbits(buf, axis=-1, bitorder="little")[..., : n * bits]
    bitmat = stream.reshape(buf.shape[:-1] + (n, bits)).astype(np.uint16)
    return (bitmat << np.arange(bits, dtype=np.uint16)).sum(axis=-1).astype(np.uint8)


# ---------------------------------------------------------------- plane helpers
def _plane_weights() -> np.ndarray:
    j = np.arange(16)[:, None]
    e = np.arange(2)[None, :]
    return (np.uint64(1) << (16 * e + j).astype(np.uint64))  # [16 j, 2 e]


def bits_to_plane_words(bits: np.ndarray) -> np.ndarray:
    """0/1 array [..., n] (n % 32 == 0) -> uint32 [..., n/32], even/odd split order."""
    b = np.asarray(bits, dtype=np.uint64)
    n = b.shape[-1]
    b = b.reshape(b.shape[:-1] + (n // 32, 16, 2))
    return (b * _plane_weights()).sum(axis=(-2, -1)).astype(np.uint32)


def plane_words_to_bits(words: np.ndarray) -> np.ndarray:
    w = np.asarray(words, dtype=np.uint64)[..., None, None]
    b = (w >> ((16 * np.arange(2)[None, :] + np.arange(16)[:, None]).astype(np.uint64))) & np.uint64(1)
    return b.reshape(words.shape[:-1] + (words.shape[-1] * 32,)).astype(np.uint8)


def codes_to_vq_words(codes: np.ndarray, bits: int = 2) -> np.ndarray:
    """Value codes [..., 16 tokens, d] -> uint32 words (dimension-major).

    2-bit: one word per dimension, token 2j + e at bit 16 e + 2 j -> [..., d].
    4-bit: two words per dimension, word w holding tokens 8 w + 2 j + e at bit 16 e + 4 j;
    all words of w = 0 first, then all of w = 1 -> [..., 2 d].
    """
    c = np.asarray(codes, dtype=np.uint64)
    d = c.shape[-1]
    if bits == 2:
        c = c.reshape(c.shape[:-2] + (8, 2, d))  # token = 2j + e
        sh = (16 * np.arange(2)[None, :] + 2 * np.arange(8)[:, None]).astype(np.uint64)[..., None]
        return (c << sh).sum(axis=(-3, -2)).astype(np.uint32)
    assert bits == 4
    c = c.reshape(c.shape[:-2] + (2, 4, 2, d))  # token = 8w + 2j + e
    sh = (16 * np.arange(2)[None, :] + 4 * np.arange(4)[:, None]).astype(np.uint64)[..., None]
    w = (c << sh).sum(axis=(-3, -2)).astype(np.uint32)  # [..., 2, d]
    return w.reshape(w.shape[:-2] + (2 * d,))


def vq_words_to_codes(words: np.ndarray, bits: int = 2) -> np.ndarray:
    if bits == 2:
        w = np.asarray(words, dtype=np.uint64)[..., None, None, :]
        sh = (16 * np.arange(2)[None, :] + 2 * np.arange(8)[:, None]).astype(np.uint64)[..., None]
        c = (w >> sh) & np.uint64(3)
        return c.reshape(words.shape[:-1] + (16, words.shape[-1])).astype(np.uint8)
    assert bits == 4
    d = words.shape[-1] // 2
    w = np.asarray(words, dtype=np.uint64).reshape(words.shape[:-1] + (2, 1, 1, d))
    sh = (16 * np.arange(2)[None, :] + 4 * np.arange(4)[:, None]).astype(np.uint64)[..., None]
    c = (w >> sh) & np.uint64(15)  # [..., 2, 4, 2, d]
    return c.reshape(words.shape[:-1] + (16, d)).astype(np.uint8)


def _u32_bytes(words: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(np.asarray(words, dtype="<u4"))
    return w.view(np.uint8).reshape(w.shape[:-1] + (w.shape[-1] * 4,))


def _f16_bytes(x: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(np.asarray(x, dtype="<f2"))
    return h.view(np.uint8).reshape(h.shape[:-1] + (h.shape[-1] * 2,))


# ---------------------------------------------------------------- main layout
def main_tile_bytes(d: int, vbits: int = 2, kbits: int = 3) -> int:
    """Key planes 2 kbits d (kbits - 1 Lloyd-Max index bits + 1 QJL bit per coordinate), value
    codes 2 vbits d, value scale/minimum 2d, two norm rows 64 B."""
    return (2 * kbits + 2 * vbits + 2) * d + 64


def main_bytes_per_token_head(d: int, vbits: int = 2, kbits: int = 3) -> float:
    return main_tile_bytes(d, vbits, kbits) / P


def main_bits(tile_bytes: int, d: int, kbits: int = None):
    """(key bits, value bits) of a main-layout tile of the given size.

    Key bits 2, 3 or 4, value bits 2 or 4.  With the key bits given, the size gives the value
    bits; without, the size alone decides for key bits 2 and 3 (sums 4..7 are distinct); in the
    one tie (4-bit keys with 2-bit values are as large as 2-bit keys with 4-bit values) the latter
    is returned, so readers of 4-bit-key tiles pass the key bits (from the codebook size).
    """
    for kb in ((kbits,) if kbits else (3, 2, 4)):
        for vbits in (2, 4):
            if main_tile_bytes(d, vbits, kb) == tile_bytes:
                return kb, vbits
    raise AssertionError((tile_bytes, d, kbits))


def main_value_bits(tile_bytes: int, d: int) -> int:
    """Value bit width of a main-layout tile of the given size."""
    return main_bits(tile_bytes, d)[1]


def pack_main_tiles(idx, sigma, vq, vs16, vmn16, nk16, nr16, vbits: int = 2, kbits: int = 3) -> np.ndarray:
    """Build main-layout tiles.

    Leading shape [..., 16 tokens]: idx, sigma, vq are [..., 16, d] uint8;
    vs16/vmn16 [..., 16, d/32] fp16; nk16/nr16 [..., 16] fp16.
    Key planes: the Lloyd-Max index bits, high bit first (kbits - 1 planes), then the QJL sign
    bits.  Returns uint8 [..., main_tile_bytes(d, vbits, kbits)].
    """
    idx = np.asarray(idx, dtype=np.uint8)
    d = idx.shape[-1]
    lead = idx.shape[:-2]
    lm_planes = [(idx >> (kbits - 2 - i)) & 1 for i in range(kbits - 1)]
    kp = [_u32_bytes(bits_to_plane_words(pl)).reshape(lead + (2 * d,)) for pl in lm_planes]
    ks = _u32_bytes(bits_to_plane_words(sigma)).reshape(lead + (2 * d,))
    vqb = _u32_bytes(codes_to_vq_words(vq, vbits))
    sm = np.stack([np.asarray(vs16, np.float16), np.asarray(vmn16, np.float16)], axis=-1)
    vsm = _f16_bytes(sm.reshape(lead + (16 * (d // 32) * 2,)))
    kn = _f16_bytes(nk16)
    rn = _f16_bytes(nr16)
    out = np.concatenate(kp + [ks, vqb, vsm, kn, rn], axis=-1)
    assert out.shape[-1] == main_tile_bytes(d, vbits, kbits)
    return out


def unpack_main_tiles(tiles: np.ndarray, d: int, kbits: int = None) -> dict:
    t = np.asarray(tiles, dtype=np.uint8)
    lead = t.shape[:-1]
    g = d // 32
    kb, vb = main_bits(t.shape[-1], d, kbits)
    o_vq = 2 * kb * d
    o_sm = o_vq + 2 * vb * d
    o_n = o_sm + 2 * d

    def words(off, nbytes):
        return np.ascontiguousarray(t[..., off:off + nbytes]).view("<u4")

    def plane(i):
        return plane_words_to_bits(words(2 * d * i, 2 * d).reshape(lead + (16, d // 32)))

    idx = np.zeros(lead + (16, d), np.int64)
    for i in range(kb - 1):
        idx = 2 * idx + plane(i)
    ks = plane(kb - 1)
    vq = vq_words_to_codes(words(o_vq, 2 * vb * d), vb)
    sm = np.ascontiguousarray(t[..., o_sm:o_sm + 2 * d]).view("<f2").reshape(lead + (16, g, 2))
    nk = np.ascontiguousarray(t[..., o_n:o_n + 32]).view("<f2")
    nr = np.ascontiguousarray(t[..., o_n + 32:o_n + 64]).view("<f2")
    return {
        "idx": idx.astype(np.uint8),
        "sigma": ks,
        "vq": vq,
        "vs": sm[..., 0].astype(np.float16),
        "vmn": sm[..., 1].astype(np.float16),
        "n_k": nk.astype(np.float16),
        "n_r": nr.astype(np.float16),
    }


# ---------------------------------------------------------------- alternate layout
def alt_key_plane_bytes(d: int, kbits: int = 8) -> int:
    """Key bytes of one alternate-layout page: the code streams and their (scale, minimum) pairs,
    or the fp16 keys alone (kbits 16)."""
    return 32 * d if kbits == 16 else 2 * kbits * d + 2 * d


def alt_tile_bytes(d: int, vbits: int = 3, kbits: int = 8) -> int:
    """One page of the alternate layout: 16 x (a dense kbits-bit stream of key codes (bytes for 8
    bits) + d/32 fp16 (scale, minimum) pairs + a dense vbits-bit stream of value indices + one fp16
    value norm); with kbits 16, 16 x (d fp16 keys + the value stream + the norm)."""
    return alt_key_plane_bytes(d, kbits) + 2 * vbits * d + 32


def alt_bytes_per_token_head(d: int, vbits: int = 3, kbits: int = 8) -> float:
    return alt_tile_bytes(d, vbits, kbits) / P


def alt_value_bits(tile_bytes: int, d: int, kbits: int = 8) -> int:
    """Value bits of an alternate-layout tile from its size and key bits."""
    vb, rem = divmod(tile_bytes - alt_key_plane_bytes(d, kbits) - 32, 2 * d)
    assert rem == 0 and 2 <= vb <= 8, (tile_bytes, d, kbits)
    return vb


def alt_key_bits(tile_bytes: int, d: int, vbits: int) -> int:
    """Key bits of an alternate-layout tile from its size and value bits."""
    key = tile_bytes - 2 * vbits * d - 32
    if key == 32 * d:
        return 16
    kb, rem = divmod(key - 2 * d, 2 * d)
    assert rem == 0 and kb in (2, 4, 5, 8), (tile_bytes, d, vbits)
    return kb


def pack_alt_tiles(kq, ks16, kmn16, vidx, nv16, vbits: int = 3, kbits: int = 8) -> np.ndarray:
    """kq [..., 16, d] (kbits-bit codes, or the fp16 keys for kbits 16); ks16/kmn16 [..., 16, d/32]
    (unused for kbits 16); vidx [..., 16, d] (vbits-bit); nv16 [..., 16]."""
    vidx = np.asarray(vidx, dtype=np.uint8)
    d = vidx.shape[-1]
    lead = vidx.shape[:-2]
    if kbits == 16:
        keys = [_f16_bytes(np.asarray(kq, np.float16).reshape(lead + (16 * d,)))]
    else:
        kq = np.asarray(kq, dtype=np.uint8)
        kqb = pack_rows(kq, kbits).reshape(lead + (16 * kbits * d // 8,))
        sm = np.stack([np.asarray(ks16, np.float16), np.asarray(kmn16, np.float16)], axis=-1)
        keys = [kqb, _f16_bytes(sm.reshape(lead + (16 * (d // 32) * 2,)))]
    vi = pack_rows(vidx, vbits).reshape(lead + (16 * vbits * d // 8,))
    vn = _f16_bytes(nv16)
    out = np.concatenate(keys + [vi, vn], axis=-1)
    assert out.shape[-1] == alt_tile_bytes(d, vbits, kbits)
    return out


def unpack_alt_tiles(tiles: np.ndarray, d: int, vbits: int = None) -> dict:
    """Fields of alternate-layout tiles.  Without vbits the keys are taken as 8-bit and the value
    bits are read off the size; with vbits (the codebook's) the key bits are read off the size.
    Tiles with fp16 keys give the field "k16" in place of "kq", "ks" and "kmn"."""
    t = np.asarray(tiles, dtype=np.uint8)
    lead = t.shape[:-1]
    g = d // 32
    if vbits is None:
        kb, vb = 8, alt_value_bits(t.shape[-1], d)
    else:
        kb, vb = alt_key_bits(t.shape[-1], d, vbits), vbits
    o_vi = alt_key_plane_bytes(d, kb)
    o_n = o_vi + 2 * vb * d
    vi = unpack_rows(t[..., o_vi:o_n].reshape(lead + (16, vb * d // 8)), d, vb)
    nv = np.ascontiguousarray(t[..., o_n:o_n + 32]).view("<f2")
    if kb == 16:
        k16 = np.ascontiguousarray(t[..., :o_vi]).view("<f2").reshape(lead + (16, d))
        return {"k16": k16.astype(np.float16), "vidx": vi, "n_v": nv.astype(np.float16)}
    o_sm = 2 * kb * d
    kq = unpack_rows(t[..., :o_sm].reshape(lead + (16, kb * d // 8)), d, kb)
    sm = np.ascontiguousarray(t[..., o_sm:o_vi]).view("<f2").reshape(lead + (16, g, 2))
    return {
        "kq": kq.copy(),
        "ks": sm[..., 0].astype(np.float16),
        "kmn": sm[..., 1].astype(np.float16),
        "vidx": vi,
        "n_v": nv.astype(np.float16),
    }


# ---------------------------------------------------------------- pools
def tile_addr(block_table: np.ndarray, b: int, pos: np.ndarray):
    """(physical block, slot) for token positions ``pos`` of sequence b."""
    pos = np.asarray(pos)
    return block_table[b, pos // P], pos % P
