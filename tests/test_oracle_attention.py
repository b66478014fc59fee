"""Pins for the oracle's decode attention."""
import numpy as np
import pytest
import torch

import synth
from oracle import attention, cache, codebook, layout, quant, rng, rotation


def _setup_main(seed, bsz, hkv, n_rep, d, lengths, shuffled=True):
    sg = rng.signs(seed, d)
    c, _ = codebook.lloyd_max(d, 2)
    s = rng.gaussian_matrix(seed, d, d)
    lmax = max(lengths)
    t_all = ((lmax + 15) // 16) * 16
    k, v = synth.kv_main(seed, bsz, hkv, t_all, d)
    max_blocks = t_all // 16
    bt = synth.block_table(seed, bsz, max_blocks, shuffled)
    pool = np.zeros((bsz * max_blocks, hkv, layout.main_tile_bytes(d)), np.uint8)
    n_c = np.zeros(bsz, np.int64)
    n_b = np.zeros(bsz, np.int64)
    ring_k = np.zeros((bsz, hkv, 128, d), np.float16)
    ring_v = np.zeros_like(ring_k)
    for b, L in enumerate(lengths):
        nc, nb = cache.ring_split(L)
        n_c[b], n_b[b] = nc, nb
        if nc:
            cache.encode_main_range(pool, bt[b:b + 1], 0, k[b:b + 1, :, :nc], v[b:b + 1, :, :nc], sg, c, s)
        ring_k[b, :, :nb] = k[b, :, nc:nc + nb]
        ring_v[b, :, :nb] = v[b, :, nc:nc + nb]
    q = synth.queries(seed, bsz, hkv * n_rep, d)
    return dict(q=q, pool=pool, bt=bt, n_c=n_c, n_b=n_b, ring_k=ring_k, ring_v=ring_v, sg=sg, c=c, s=s,
                hkv=hkv, k=k, v=v)


def test_estimator_form_equals_bruteforce_softmax():
    e = _setup_main(1, 2, 2, 3, 64, [200, 37])
    args = (e["q"], e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], e["sg"], e["c"], e["s"], e["hkv"])
    fast = attention.decode_main(*args)
    brute = attention.decode_main_bruteforce(*args)
    assert np.allclose(fast, brute, rtol=0, atol=1e-12)


def test_ring_only_is_exact_attention_and_matches_torch_sdpa():
    e = _setup_main(2, 2, 2, 4, 128, [100, 128])
    out = attention.decode_main(e["q"], e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"],
                                e["sg"], e["c"], e["s"], e["hkv"])
    for b, L in enumerate([100, 128]):
        q = torch.tensor(e["q"][b:b + 1].astype(np.float64))[:, :, None, :]
        k = torch.tensor(e["k"][b:b + 1, :, :L].astype(np.float64)).repeat_interleave(4, dim=1)
        v = torch.tensor(e["v"][b:b + 1, :, :L].astype(np.float64)).repeat_interleave(4, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v)[:, :, 0, :].numpy()
        assert np.allclose(out[b:b + 1], ref, rtol=1e-10, atol=1e-10)


def test_gqa_head_mapping_matches_repeated_kv():
    """Query head h reads KV head h // n_rep: compare with per-head single-head decodes."""
    e = _setup_main(3, 1, 2, 2, 64, [300])
    full = attention.decode_main(e["q"], e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"],
                                 e["sg"], e["c"], e["s"], 2)
    for h in range(4):
        g = h // 2
        one = attention.decode_main(e["q"][:, h:h + 1], e["pool"][:, g:g + 1], e["bt"], e["n_c"],
                                    e["ring_k"][:, g:g + 1], e["ring_v"][:, g:g + 1], e["n_b"],
                                    e["sg"], e["c"], e["s"], 1)
        assert np.allclose(one[:, 0], full[:, h], atol=1e-14)


def test_compressed_logits_track_exact_logits():
    """Sanity of the encode chain: estimated logits correlate with exact fp16 logits."""
    e = _setup_main(4, 1, 2, 4, 128, [1024])
    f = cache.read_main(e["pool"], e["bt"], 0, 896, 128)
    q = e["q"][0, 0].astype(np.float64)
    est = quant.inner_product_estimate(q, f["n_k"][0], f["idx"][0], f["n_r"][0], f["sigma"][0], e["sg"], e["c"], e["s"])
    exact = e["k"][0, 0, :896].astype(np.float64) @ q
    assert np.corrcoef(est, exact)[0, 1] > 0.85


@pytest.mark.parametrize("vbits,kbits", [(2, 8), (3, 8), (4, 8), (3, 4), (3, 5), (3, 2), (2, 2), (5, 8), (8, 8)])
def test_alt_layout_decode_matches_torch_sdpa_on_dequantised_cache(vbits, kbits):
    d, hkv, n_rep = 64, 2, 1
    sg = rng.signs(5, d)
    c3, _ = codebook.lloyd_max(d, vbits)
    k, v = synth.kv_alt(5, 1, hkv, 64, d)
    bt = synth.block_table(5, 1, 4, True)
    pool = np.zeros((4, hkv, layout.alt_tile_bytes(d, vbits, kbits)), np.uint8)
    cache.encode_alt_range(pool, bt, 0, k, v, sg, c3)
    q = synth.queries(5, 1, hkv * n_rep, d)
    out = attention.decode_alt(q, pool, bt, np.array([64]), None, None, None, sg, c3, hkv)
    kq, ks, kmn = quant.encode_alt_keys(k, bits=kbits)
    assert kq.max() == (1 << kbits) - 1
    khat = quant.group_dequant(kq, ks, kmn, 32)
    venc = quant.encode_alt_values(v, sg, c3)
    # butterfly pulled out: sum_t p_t * unrotate(x_t) == unrotate(sum_t p_t x_t)
    vr = venc["n_v"].astype(np.float64)[..., None] * c3[venc["idx"]]
    vhat = rotation.unrotate(vr, sg)
    p = np.random.default_rng(0).random(64)
    assert np.allclose(p @ vhat[0, 0], rotation.unrotate(p @ vr[0, 0], sg), atol=1e-12)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q.astype(np.float64))[:, :, None, :], torch.tensor(khat), torch.tensor(vhat))[:, :, 0, :]
    assert np.allclose(out, ref.numpy(), atol=1e-10)


@pytest.mark.parametrize("vbits", [2, 3, 4])
def test_alt_layout_fp16_keys_decode_matches_torch_sdpa(vbits):
    # keys kept as fp16, values rotated and Lloyd-Max quantised ("TurboQuant-MLX overview", usage
    # paths: the V-only cache): the logits are the exact q k / sqrt(d) of the fp16 keys
    d, hkv, n_rep = 64, 2, 2
    sg = rng.signs(7, d)
    c, _ = codebook.lloyd_max(d, vbits)
    k, v = synth.kv_alt(7, 1, hkv, 96, d)
    bt = synth.block_table(7, 1, 6, True)
    pool = np.zeros((6, hkv, layout.alt_tile_bytes(d, vbits, 16)), np.uint8)
    cache.encode_alt_range(pool, bt, 0, k, v, sg, c)
    q = synth.queries(7, 1, hkv * n_rep, d)
    out = attention.decode_alt(q, pool, bt, np.array([96]), None, None, None, sg, c, hkv)
    venc = quant.encode_alt_values(v, sg, c)
    vhat = quant.dequant_alt_values(venc["idx"], venc["n_v"], sg, c)
    kk = torch.tensor(k.astype(np.float64)).repeat_interleave(n_rep, dim=1)
    vv = torch.tensor(vhat).repeat_interleave(n_rep, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q.astype(np.float64))[:, :, None, :], kk, vv)[:, :, 0, :]
    assert np.allclose(out, ref.numpy(), atol=1e-10)


def test_empty_and_zero_key_cases():
    e = _setup_main(6, 2, 1, 2, 64, [1, 130])
    # zero a compressed key: its logit becomes exactly 0
    out = attention.decode_main(e["q"], e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"],
                                e["sg"], e["c"], e["s"], 1)
    assert np.all(np.isfinite(out))
    # length-1 sequence attends to its single ring token: output equals that value
    assert np.allclose(out[0], e["v"][0, 0, 0].astype(np.float64)[None, :], atol=1e-12)
