"""Parity at the benchmark workloads' full sizes (GPU), on sampled outputs.

Every decode step here runs the whole batch, with the benchmark's launch configuration, through
the C ABI. The oracle cannot decode a whole 32K-131K batch in seconds, so for each workload:

* a few sequences are encoded by the oracle (their pages are uploaded) and the rest by
  ``tq_encode_flush`` on the GPU; the oracle checks the decode outputs of its own sequences
  only, so no oracle input ever comes from the CUDA path;
* a sample of pages that the GPU encoded is compared with the oracle's encoding of the same
  tokens (value planes bit-exact, Lloyd-Max / QJL bits away from decision boundaries, norms
  within 1 fp16 ulp).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_cases import (MARGIN, allclose_report, alt_fields, main_fields, make_ctx, near_boundary, to_dev)
from oracle import attention, cache, layout, quant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from kv_cache_quantization_tq_gb300.build import build

    build()
    import kv_cache_quantization_tq_gb300 as tq


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bench_max_ctx(lengths):
    # bench.py sizes the workspace for the prefix plus warm-up, timed and end-to-end steps
    return ((max(lengths) + 3 + 64 + 64 + 15) // 16) * 16


def _run_main(seed, hq, hkv, lengths, oracle_seqs, shuffled=True, n_sample_pages=24, paths=(None,)):
    d = 128
    bsz = len(lengths)
    ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, seed)
    max_ctx = _bench_max_ctx(lengths)
    max_blocks = max_ctx // 16 + 8
    bt = synth.block_table(seed, bsz, max_blocks, shuffled)
    nblk = bsz * max_blocks
    tile = layout.main_tile_bytes(d)
    pool = torch.zeros((nblk, hkv, tile), dtype=torch.uint8, device="cuda")
    bt_d = to_dev(bt)
    ring_k = np.zeros((bsz, hkv, 128, d), np.float16)
    ring_v = np.zeros_like(ring_k)
    n_c = np.zeros(bsz, np.int32)
    n_b = np.zeros(bsz, np.int32)
    oracle_pools = {}
    rng = np.random.default_rng(seed)
    checked_pages = 0
    for b, L in enumerate(lengths):
        nc, nb = cache.ring_split(L)
        n_c[b], n_b[b] = nc, nb
        k, v = synth.kv_main(seed, 1, hkv, L, d, layer=b)
        ring_k[b, :, :nb] = k[0, :, nc:nc + nb]
        ring_v[b, :, :nb] = v[0, :, nc:nc + nb]
        if not nc:
            continue
        if b in oracle_seqs:
            p = np.zeros((nblk, hkv, tile), np.uint8)
            cache.encode_main_range(p, bt[b:b + 1], 0, k[:, :, :nc], v[:, :, :nc], s, c, sk)
            blocks = bt[b, :nc // 16]
            pool[torch.from_numpy(blocks.astype(np.int64)).cuda()] = torch.from_numpy(p[blocks]).cuda()
            oracle_pools[b] = p
        else:
            ctx.encode_flush(to_dev(k), to_dev(v), to_dev(np.zeros(1, np.int32)), bt_d[b:b + 1], pool, n_tokens=nc)
            # sampled pages of this GPU-encoded sequence against the oracle's encoding of the same tokens
            pages = rng.choice(nc // 16, size=min(n_sample_pages // max(1, bsz - len(oracle_seqs)) + 1, nc // 16),
                               replace=False)
            got = pool[torch.from_numpy(bt[b, pages].astype(np.int64)).cuda()].cpu().numpy()
            for i, pg in enumerate(pages):
                kk = k[:, :, pg * 16:(pg + 1) * 16]
                vv = v[:, :, pg * 16:(pg + 1) * 16]
                ref = np.zeros((1, hkv, tile), np.uint8)
                enc = cache.encode_main_range(ref, np.zeros((1, 1), np.int32), 0, kk, vv, s, c, sk)
                fo, fg = main_fields(ref[0], d), main_fields(got[i], d)
                assert np.array_equal(fg["v_bytes"], fo["v_bytes"])
                near = near_boundary(enc["y"][0], c)
                idx_diff = fg["idx"] != fo["idx"]
                assert not (idx_diff & ~near).any()
                tok_diff = idx_diff.any(axis=-1)
                assert not ((fg["sigma"] != fo["sigma"]) & ~(np.abs(enc["z"][0]) < MARGIN) & ~tok_diff[..., None]).any()
                assert np.max(np.abs(fg["kn"].astype(np.int32) - fo["kn"].astype(np.int32))) <= 1
                checked_pages += 1
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    q = synth.queries(seed, bsz, hq, d)
    refs = {}
    for b in oracle_seqs:
        p = oracle_pools.get(b, np.zeros((nblk, hkv, tile), np.uint8))
        refs[b] = attention.decode_main(q[b:b + 1], p, bt[b:b + 1], n_c[b:b + 1], ring_k[b:b + 1], ring_v[b:b + 1],
                                        n_b[b:b + 1], s, c, sk, hkv)
    for path in paths:  # None: the default path; else a TQ_DECODE_* value
        if path is not None:
            ctx.set_decode_path(path)
        out = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
        ws = torch.empty(ctx.workspace_size(bsz, max_ctx), dtype=torch.uint8, device="cuda")
        ctx.decode_attention(to_dev(q), pool, bt_d, to_dev(n_c), to_dev(ring_k), to_dev(ring_v), to_dev(n_b),
                             max_ctx, out, ws)
        got = out.cpu().numpy()
        assert ctx.device_errors() == 0
        assert np.all(np.isfinite(got))
        for b in oracle_seqs:
            ok, maxerr, nbad = allclose_report(got[b:b + 1], refs[b])
            assert ok, f"path {path}, sequence {b}: max abs err {maxerr}, {nbad} outside tolerance"
    return checked_pages


def test_qwen25_7b_b8_32k_shuffled_pages():
    """Batch 8, 28 q / 4 KV heads, 32768 tokens each, shuffled 16-token pages; the default decoder
    and the tcgen05 score path on the same cache."""
    assert _run_main(0, 28, 4, [32768] * 8, oracle_seqs={0, 5},
                     paths=(None, tq.TQ_DECODE_TCGEN05)) > 0


def test_qwen3_06b_32k_two_layers():
    """Batch 1, 16 q / 4 KV heads, 32768-token prefix; two layers (two table seeds)."""
    for layer in range(2):
        _run_main(layer, 16, 4, [32768], oracle_seqs={0}, shuffled=False, n_sample_pages=8)


def test_qwen25_32b_ragged_batch16():
    """Batch 16, 40 q / 8 KV heads, lengths U[1024, 131072] (seed 7), shuffled pages."""
    lengths = [int(x) for x in synth.ragged_lengths(7, 16, 1024, 131072)]
    short, longest = int(np.argmin(lengths)), int(np.argmax(lengths))
    # the longest sequence has the most split-K chunk slots of the plan
    _run_main(7, 40, 8, lengths, oracle_seqs={short, 3, longest})


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_alt_layout_65536_head_dim_sweep(d):
    """Alternate layout, 8 q / 8 KV heads, batch 4, 65536 tokens, no ring; every KV head of sequence 1
    checked."""
    hq = hkv = 8
    bsz, L, seed = 4, 65536, 11
    ctx, c3, s, _ = make_ctx(tq, False, d, hq, hkv, seed)
    max_blocks = L // 16
    bt = synth.block_table(seed, bsz, max_blocks, False)
    tile = layout.alt_tile_bytes(d)
    pool = torch.zeros((bsz * max_blocks, hkv, tile), dtype=torch.uint8, device="cuda")
    check_b = 1
    heads = list(range(hkv))  # oracle-checked KV heads of the checked sequence
    p_or = None
    for b in range(bsz):
        k, v = synth.kv_alt(seed, 1, hkv, L, d, layer=b)
        if b == check_b:
            p_or = np.zeros((bsz * max_blocks, len(heads), tile), np.uint8)
            cache.encode_alt_range(p_or, bt[b:b + 1], 0, k[:, heads], v[:, heads], s, c3)
            kv_b = (k, v)
        ctx.encode_flush(to_dev(k), to_dev(v), to_dev(np.zeros(1, np.int32)), to_dev(bt[b:b + 1]), pool)
    # GPU-encoded tiles of the checked heads: key planes bit-exact vs the oracle, value indices
    # away from boundaries
    blocks = bt[check_b]
    sample = blocks[:: max(1, len(blocks) // 32)]
    g_tiles = pool[torch.from_numpy(sample.astype(np.int64)).cuda()].cpu().numpy()[:, heads]
    o_tiles = p_or[sample]
    fo, fg = alt_fields(o_tiles, d), alt_fields(g_tiles, d)
    assert np.array_equal(fg["k_bytes"], fo["k_bytes"])
    k, v = kv_b
    pages = (np.arange(len(blocks))[:: max(1, len(blocks) // 32)])
    yv = []
    for pg in pages:
        yv.append(quant.encode_alt_values(v[0, heads, pg * 16:(pg + 1) * 16], s, c3)["y"])
    near = near_boundary(np.stack(yv), c3)
    assert not ((fg["vidx"] != fo["vidx"]) & ~near).any()
    # decode the whole batch from the GPU pool, but check the checked sequence on a pool whose
    # checked heads hold the oracle's pages
    pool_chk = pool.clone()
    for i, h in enumerate(heads):
        pool_chk[torch.from_numpy(blocks.astype(np.int64)).cuda(), h] = torch.from_numpy(p_or[blocks, i]).cuda()
    q = synth.queries(seed, bsz, hq, d)
    n_c = np.full(bsz, L, np.int32)
    out = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(bsz, L), dtype=torch.uint8, device="cuda")
    ctx.decode_attention(to_dev(q), pool_chk, to_dev(bt), to_dev(n_c), None, None, None, L, out, ws)
    got = out.cpu().numpy()
    assert ctx.device_errors() == 0
    ref = attention.decode_alt(q[check_b:check_b + 1, heads], p_or, bt[check_b:check_b + 1], n_c[check_b:check_b + 1],
                               None, None, None, s, c3, len(heads))
    ok, maxerr, nbad = allclose_report(got[check_b, heads][None], ref)
    assert ok, f"max abs err {maxerr}, {nbad} bad"
