"""Pins for the oracle's prefill materialisation (dense history from the compressed pool)."""
import numpy as np
import pytest

import synth
from oracle import attention, cache, codebook, layout, rng

from test_oracle_attention import _setup_main


def _attend(q16, k, v, n_kv):
    """Plain float64 softmax attention of q [Hq, d] over k, v [Hkv, T, d]."""
    q = np.asarray(q16, np.float64)
    hq, d = q.shape
    n_rep = hq // n_kv
    out = np.zeros((hq, d))
    for h in range(hq):
        g = h // n_rep
        z = k[g] @ q[h] / np.sqrt(d)
        w = np.exp(z - z.max())
        out[h] = w @ v[g] / w.sum()
    return out


def test_main_materialised_history_reproduces_the_decode_estimator():
    # attention over (k^, v^) is the decode step computed from the packed bits (estimator form)
    e = _setup_main(3, 2, 2, 3, 64, [300, 160])
    args = (e["q"], e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], e["sg"], e["c"], e["s"], e["hkv"])
    ref = attention.decode_main(*args)
    for b in range(2):
        k, v = cache.materialize_main(e["pool"], e["bt"], b, int(e["n_c"][b]), e["ring_k"], e["ring_v"],
                                      int(e["n_b"][b]), e["sg"], e["c"], e["s"], 64)
        assert k.shape == (2, 300 if b == 0 else 160, 64)
        assert np.allclose(_attend(e["q"][b], k, v, e["hkv"]), ref[b], rtol=0, atol=1e-12)


def test_main_materialised_rows_keep_ring_exact_and_values_within_half_a_step():
    e = _setup_main(4, 1, 2, 1, 128, [1000])
    nc, nb = int(e["n_c"][0]), int(e["n_b"][0])
    k, v = cache.materialize_main(e["pool"], e["bt"], 0, nc, e["ring_k"], e["ring_v"], nb, e["sg"], e["c"], e["s"], 128)
    # ring rows are the exact fp16 tokens
    assert np.array_equal(k[:, nc:], e["k"][0, :, nc:nc + nb].astype(np.float64))
    assert np.array_equal(v[:, nc:], e["v"][0, :, nc:nc + nb].astype(np.float64))
    # the asymmetric quantiser: |v^ - v| <= s/2 (plus rounding), s = (max - min)/3 per group of 32
    v0 = e["v"][0, :, :nc].astype(np.float64).reshape(2, nc, 4, 32)
    step = (v0.max(-1) - v0.min(-1)) / 3.0
    err = np.abs(v[:, :nc].reshape(2, nc, 4, 32) - v0)
    assert np.all(err <= step[..., None] * (0.5 + 2e-3) + 1e-6)
    # keys: the reconstruction is unbiased in the sketch, so on average it points along k
    k0 = e["k"][0, :, :nc].astype(np.float64)
    cos = np.sum(k[:, :nc] * k0, -1) / (np.linalg.norm(k[:, :nc], axis=-1) * np.linalg.norm(k0, axis=-1))
    assert cos.mean() > 0.8


@pytest.mark.parametrize("vbits,kbits", [(2, 8), (3, 8), (4, 8), (3, 4), (3, 5), (3, 2), (2, 2), (6, 8), (8, 4)])
def test_alt_materialised_history_reproduces_the_decode(vbits, kbits):
    seed, d, hkv, bsz = 5, 64, 2, 2
    sg = rng.signs(seed, d)
    c3, _ = codebook.lloyd_max(d, vbits)
    lengths = [160, 96]
    k, v = synth.kv_alt(seed, bsz, hkv, 160, d)
    bt = synth.block_table(seed, bsz, 10, True)
    pool = np.zeros((bsz * 10, hkv, layout.alt_tile_bytes(d, vbits, kbits)), np.uint8)
    for b, L in enumerate(lengths):
        cache.encode_alt_range(pool, bt[b:b + 1], 0, k[b:b + 1, :, :L], v[b:b + 1, :, :L], sg, c3)
    q = synth.queries(seed, bsz, hkv, d)
    n_c = np.array(lengths)
    ref = attention.decode_alt(q, pool, bt, n_c, None, None, None, sg, c3, hkv)
    for b, L in enumerate(lengths):
        kk, vv = cache.materialize_alt(pool, bt, b, L, None, None, 0, sg, c3, d)
        assert np.allclose(_attend(q[b], kk, vv, hkv), ref[b], rtol=0, atol=1e-12)
        # keys: (2^kbits - 1)-step affine codes per block of 32, error at most half a step
        k0 = k[b, :, :L].astype(np.float64).reshape(hkv, L, d // 32, 32)
        step = (k0.max(-1) - k0.min(-1)) / ((1 << kbits) - 1.0)
        assert np.all(np.abs(kk.reshape(hkv, L, d // 32, 32) - k0) <= step[..., None] * (0.5 + 2e-3) + 1e-6)


def test_alt_materialised_fp16_keys_are_the_inputs():
    seed, d, hkv, vbits = 9, 64, 2, 3
    sg = rng.signs(seed, d)
    c3, _ = codebook.lloyd_max(d, vbits)
    k, v = synth.kv_alt(seed, 1, hkv, 64, d)
    bt = synth.block_table(seed, 1, 4, True)
    pool = np.zeros((4, hkv, layout.alt_tile_bytes(d, vbits, 16)), np.uint8)
    cache.encode_alt_range(pool, bt, 0, k, v, sg, c3)
    kk, vv = cache.materialize_alt(pool, bt, 0, 64, None, None, 0, sg, c3, d)
    assert np.array_equal(kk, k[0].astype(np.float64))  # no key quantisation at all
    q = synth.queries(seed, 1, hkv, d)
    ref = attention.decode_alt(q, pool, bt, np.array([64]), None, None, None, sg, c3, hkv)
    assert np.allclose(_attend(q[0], kk, vv, hkv), ref[0], rtol=0, atol=1e-12)


def test_main_layout_with_4bit_values():
    # the same pins with 4-bit value codes (15 levels per group of 32)
    seed, d, hkv, n_rep = 6, 64, 2, 2
    sg = rng.signs(seed, d)
    c, _ = codebook.lloyd_max(d, 2)
    s = rng.gaussian_matrix(seed, d, d)
    lengths = [300, 129]
    k, v = synth.kv_main(seed, 2, hkv, 304, d)
    bt = synth.block_table(seed, 2, 19, True)
    pool = np.zeros((38, hkv, layout.main_tile_bytes(d, 4)), np.uint8)
    ring_k = np.zeros((2, hkv, 128, d), np.float16)
    ring_v = np.zeros_like(ring_k)
    n_c, n_b = np.zeros(2, np.int64), np.zeros(2, np.int64)
    for b, L in enumerate(lengths):
        nc, nb = cache.ring_split(L)
        n_c[b], n_b[b] = nc, nb
        cache.encode_main_range(pool, bt[b:b + 1], 0, k[b:b + 1, :, :nc], v[b:b + 1, :, :nc], sg, c, s)
        ring_k[b, :, :nb] = k[b, :, nc:nc + nb]
        ring_v[b, :, :nb] = v[b, :, nc:nc + nb]
    q = synth.queries(seed, 2, hkv * n_rep, d)
    ref = attention.decode_main(q, pool, bt, n_c, ring_k, ring_v, n_b, sg, c, s, hkv)
    brute = attention.decode_main_bruteforce(q, pool, bt, n_c, ring_k, ring_v, n_b, sg, c, s, hkv)
    assert np.allclose(ref, brute, rtol=0, atol=1e-12)
    for b in range(2):
        nc, nb = int(n_c[b]), int(n_b[b])
        kk, vv = cache.materialize_main(pool, bt, b, nc, ring_k, ring_v, nb, sg, c, s, d)
        assert np.allclose(_attend(q[b], kk, vv, hkv), ref[b], rtol=0, atol=1e-12)
        v0 = v[b, :, :nc].astype(np.float64).reshape(hkv, nc, d // 32, 32)
        step = (v0.max(-1) - v0.min(-1)) / 15.0
        err = np.abs(vv[:, :nc].reshape(hkv, nc, d // 32, 32) - v0)
        assert np.all(err <= step[..., None] * (0.5 + 2e-3) + 1e-6)
        # 4-bit codes are finer than 2-bit ones: mean error well under the 2-bit half step
        assert err.mean() < (step[..., None] * 15 / 3 * 0.25).mean()


def test_main_layout_with_2bit_keys():
    # 1-bit Lloyd-Max index (centroids +-E|x|) plus the QJL bit: same estimator and reconstruction pins
    seed, d, hkv, n_rep = 8, 64, 2, 3
    sg = rng.signs(seed, d)
    c, _ = codebook.lloyd_max(d, 1)
    s = rng.gaussian_matrix(seed, d, d)
    lengths = [280, 140]
    k, v = synth.kv_main(seed, 2, hkv, 288, d)
    bt = synth.block_table(seed, 2, 18, True)
    pool = np.zeros((36, hkv, layout.main_tile_bytes(d, 2, 2)), np.uint8)
    ring_k = np.zeros((2, hkv, 128, d), np.float16)
    ring_v = np.zeros_like(ring_k)
    n_c, n_b = np.zeros(2, np.int64), np.zeros(2, np.int64)
    for b, L in enumerate(lengths):
        nc, nb = cache.ring_split(L)
        n_c[b], n_b[b] = nc, nb
        cache.encode_main_range(pool, bt[b:b + 1], 0, k[b:b + 1, :, :nc], v[b:b + 1, :, :nc], sg, c, s)
        ring_k[b, :, :nb] = k[b, :, nc:nc + nb]
        ring_v[b, :, :nb] = v[b, :, nc:nc + nb]
    q = synth.queries(seed, 2, hkv * n_rep, d)
    ref = attention.decode_main(q, pool, bt, n_c, ring_k, ring_v, n_b, sg, c, s, hkv)
    brute = attention.decode_main_bruteforce(q, pool, bt, n_c, ring_k, ring_v, n_b, sg, c, s, hkv)
    assert np.allclose(ref, brute, rtol=0, atol=1e-12)
    f = cache.read_main(pool, bt, 0, int(n_c[0]), d)
    assert set(np.unique(f["idx"])) <= {0, 1}
    for b in range(2):
        kk, vv = cache.materialize_main(pool, bt, b, int(n_c[b]), ring_k, ring_v, int(n_b[b]), sg, c, s, d)
        assert np.allclose(_attend(q[b], kk, vv, hkv), ref[b], rtol=0, atol=1e-12)


def test_main_layout_with_4bit_keys():
    # 3-bit Lloyd-Max index (8 centroids) plus the QJL bit; the readers take the key width from
    # the codebook (the tile size alone would not tell it from 2-bit keys with 4-bit values)
    seed, d, hkv, n_rep = 9, 64, 2, 2
    sg = rng.signs(seed, d)
    c, _ = codebook.lloyd_max(d, 3)
    s = rng.gaussian_matrix(seed, d, d)
    lengths = [300, 150]
    k, v = synth.kv_main(seed, 2, hkv, 304, d)
    bt = synth.block_table(seed, 2, 19, True)
    pool = np.zeros((38, hkv, layout.main_tile_bytes(d, 2, 4)), np.uint8)
    ring_k = np.zeros((2, hkv, 128, d), np.float16)
    ring_v = np.zeros_like(ring_k)
    n_c, n_b = np.zeros(2, np.int64), np.zeros(2, np.int64)
    for b, L in enumerate(lengths):
        nc, nb = cache.ring_split(L)
        n_c[b], n_b[b] = nc, nb
        cache.encode_main_range(pool, bt[b:b + 1], 0, k[b:b + 1, :, :nc], v[b:b + 1, :, :nc], sg, c, s)
        ring_k[b, :, :nb] = k[b, :, nc:nc + nb]
        ring_v[b, :, :nb] = v[b, :, nc:nc + nb]
    q = synth.queries(seed, 2, hkv * n_rep, d)
    ref = attention.decode_main(q, pool, bt, n_c, ring_k, ring_v, n_b, sg, c, s, hkv)
    brute = attention.decode_main_bruteforce(q, pool, bt, n_c, ring_k, ring_v, n_b, sg, c, s, hkv)
    assert np.allclose(ref, brute, rtol=0, atol=1e-12)
    f = cache.read_main(pool, bt, 0, int(n_c[0]), d, 4)
    assert f["idx"].max() > 3  # all eight cells in use
    for b in range(2):
        kk, vv = cache.materialize_main(pool, bt, b, int(n_c[b]), ring_k, ring_v, int(n_b[b]), sg, c, s, d)
        assert np.allclose(_attend(q[b], kk, vv, hkv), ref[b], rtol=0, atol=1e-12)
    # finer keys: the Lloyd-Max part alone is closer to the rotated key than with the 2-bit index
    from oracle import quant
    y = quant.encode_keys(k[0, :, :256], sg, c, s)["y"]
    c2, _ = codebook.lloyd_max(d, 2)
    e3 = np.mean((y - c[quant.assign(y, quant.boundaries_of(c))]) ** 2)
    e2 = np.mean((y - c2[quant.assign(y, quant.boundaries_of(c2))]) ** 2)
    assert e3 < 0.4 * e2
