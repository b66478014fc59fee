"""CUDA path vs the CPU oracle, element by element, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import synth
from gpu_cases import (MARGIN, allclose_report, alt_fields, build_alt_cache, build_main_cache, main_fields, make_ctx,
                       near_boundary, tile_index, to_dev)
from oracle import attention, cache, layout, quant

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from kv_cache_quantization_tq_gb300.build import build

    build()
    import kv_cache_quantization_tq_gb300 as tq
else:  # collected on CPU-only hosts, deselected by -m "not gpu"
    tq = None


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


# ====================================================================== encode
def _encode_main_both(d, hkv, n_tok, starts, seed, src_extra=0, value_bits=2, key_bits=3):
    bsz = len(starts)
    ctx, c, s, sk = make_ctx(tq, True, d, hkv, hkv, seed, value_bits=value_bits, key_bits=key_bits)
    k, v = synth.kv_main(seed, bsz, hkv, n_tok + src_extra, d)
    k[0, 0, 3] = 0  # a zero key
    v[0, 0, 5, :32] = np.float16(0.75)  # a constant value group (scale 0)
    max_blocks = (max(starts) + n_tok) // 16 + 2
    bt = synth.block_table(seed, bsz, max_blocks, True)
    nblk = bsz * max_blocks
    pool_o = np.zeros((nblk, hkv, layout.main_tile_bytes(d, value_bits, key_bits)), np.uint8)
    encs = []
    for b in range(bsz):
        encs.append(cache.encode_main_range(pool_o, bt[b:b + 1], starts[b], k[b:b + 1, :, :n_tok], v[b:b + 1, :, :n_tok],
                                            s, c, sk))
    pool_g = torch.zeros(pool_o.shape, dtype=torch.uint8, device="cuda")
    ctx.encode_flush(to_dev(k), to_dev(v), to_dev(np.array(starts, np.int32)), to_dev(bt), pool_g, n_tokens=n_tok)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    return ctx, pool_o, pool_g.cpu().numpy(), encs, bt, c


def _compare_main(pool_o, pool_g, encs, bt, starts, n_tok, d, c):
    blocks = tile_index(bt, starts, n_tok)  # [B, pages]
    written = np.zeros(pool_o.shape[0], bool)
    written[blocks.ravel()] = True
    assert np.array_equal(pool_g[~written], pool_o[~written])  # untouched pages stay untouched
    kb = len(c).bit_length()  # key bits: Lloyd-Max index bits + the QJL bit
    fo = main_fields(pool_o[blocks], d, kb)  # [B, pages, Hkv, 16, ...]
    fg = main_fields(pool_g[blocks], d, kb)
    # value planes: bit-exact
    assert np.array_equal(fg["v_bytes"], fo["v_bytes"])
    npg = n_tok // 16
    hkv = pool_o.shape[1]
    y = np.stack([e["y"][0] for e in encs])  # [B, Hkv, T, d]
    z = np.stack([e["z"][0] for e in encs])
    y = y.reshape(len(starts), hkv, npg, 16, d).transpose(0, 2, 1, 3, 4)
    z = z.reshape(len(starts), hkv, npg, 16, d).transpose(0, 2, 1, 3, 4)
    near = near_boundary(y, c)
    idx_diff = fg["idx"] != fo["idx"]
    assert not (idx_diff & ~near).any(), "Lloyd-Max index differs away from a boundary"
    tok_diff = idx_diff.any(axis=-1)  # tokens whose residual legitimately differs
    sig_diff = (fg["sigma"] != fo["sigma"]) & ~(np.abs(z) < MARGIN) & ~tok_diff[..., None]
    assert not sig_diff.any(), f"QJL bits differ away from zero: {int(sig_diff.sum())}"
    assert np.max(np.abs(fg["kn"].astype(np.int32) - fo["kn"].astype(np.int32))) <= 1
    rn_d = np.abs(fg["rn"].astype(np.int32) - fo["rn"].astype(np.int32))
    assert np.max(np.where(tok_diff, 0, rn_d)) <= 1
    return int(near.sum()), int(idx_diff.sum())


@pytest.mark.parametrize("d", [128, 64, 256, 512])
def test_encode_main_parity(d):
    n_tok = 256 if d <= 128 else 128
    starts = [0, 64, 512]
    ctx, pool_o, pool_g, encs, bt, c = _encode_main_both(d, 2, n_tok, starts, seed=d)
    _compare_main(pool_o, pool_g, encs, bt, starts, n_tok, d, c)


def test_encode_main_ragged_tail_tokens():
    """n_tokens not a multiple of the CTA batch (208 = 128 + 80)."""
    ctx, pool_o, pool_g, encs, bt, c = _encode_main_both(128, 3, 208, [16, 0], seed=3, src_extra=32)
    _compare_main(pool_o, pool_g, encs, bt, [16, 0], 208, 128, c)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_encode_alt_parity(d):
    hkv, n_tok, starts, seed = 2, 96, [0, 32], 40 + d
    ctx, c3, s, _ = make_ctx(tq, False, d, hkv, hkv, seed)
    k, v = synth.kv_alt(seed, 2, hkv, n_tok, d)
    v[1, 1, 7] = 0  # zero value vector
    max_blocks = 10
    bt = synth.block_table(seed, 2, max_blocks, True)
    pool_o = np.zeros((2 * max_blocks, hkv, layout.alt_tile_bytes(d)), np.uint8)
    encs = [cache.encode_alt_range(pool_o, bt[b:b + 1], starts[b], k[b:b + 1], v[b:b + 1], s, c3) for b in range(2)]
    pool_g = torch.zeros(pool_o.shape, dtype=torch.uint8, device="cuda")
    ctx.encode_flush(to_dev(k), to_dev(v), to_dev(np.array(starts, np.int32)), to_dev(bt), pool_g)
    pool_g = pool_g.cpu().numpy()
    blocks = tile_index(bt, starts, n_tok)
    fo = alt_fields(pool_o[blocks], d)
    fg = alt_fields(pool_g[blocks], d)
    assert np.array_equal(fg["k_bytes"], fo["k_bytes"])  # affine int8 keys: bit-exact
    assert np.max(np.abs(fg["vn"].astype(np.int32) - fo["vn"].astype(np.int32))) <= 1
    y = np.stack([e["y"][0] for e in encs]).reshape(2, hkv, n_tok // 16, 16, d).transpose(0, 2, 1, 3, 4)
    near = near_boundary(y, c3)
    assert not ((fg["vidx"] != fo["vidx"]) & ~near).any()


# ====================================================================== decode
def _run_decode(ctx, e, q, hq, d, use_ring=True):
    bsz = q.shape[0]
    out = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(bsz, e["max_ctx"]), dtype=torch.uint8, device="cuda")
    ring_k = to_dev(e["ring_k"]) if use_ring else None
    ring_v = to_dev(e["ring_v"]) if use_ring else None
    n_buf = to_dev(e["n_b"]) if use_ring else None
    ctx.decode_attention(to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), ring_k, ring_v, n_buf,
                         e["max_ctx"], out, ws)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("d,hkv,n_rep,lengths", [
    (128, 4, 4, [1024]),                 # tiny single-layer decode step geometry
    (128, 2, 7, [1500, 300, 17, 128]),   # GQA 7, ragged, ring-only rows
    (128, 2, 5, [2049, 129]),            # GQA 5, one-token rings
    (128, 1, 16, [700]),                 # n_rep 16 -> two head groups
    (128, 1, 4, [300] * 80),             # 80 sequences: 4-warp CTAs at 2 per SM (8-warp grid > 1 per SM)
    (128, 3, 1, [333]),
    (64, 2, 2, [900, 1]),
    (256, 2, 3, [640]),
    (512, 1, 8, [400]),
])
def test_decode_main_parity(d, hkv, n_rep, lengths):
    seed = d + 7 * n_rep + len(lengths)
    hq = hkv * n_rep
    ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, seed)
    e = build_main_cache(seed, d, hkv, lengths, c, s, sk)
    q = synth.queries(seed, len(lengths), hq, d)
    got = _run_decode(ctx, e, q, hq, d)
    ref = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], s, c, sk, hkv)
    ok, maxerr, nbad = allclose_report(got, ref)
    assert ok, f"max abs err {maxerr}, {nbad} elements outside 2e-3 + 1e-3|ref|"


def test_decode_main_without_ring_argument():
    d, hkv, n_rep, seed = 128, 2, 4, 77
    ctx, c, s, sk = make_ctx(tq, True, d, hkv * n_rep, hkv, seed)
    e = build_main_cache(seed, d, hkv, [512, 256], c, s, sk)
    q = synth.queries(seed, 2, hkv * n_rep, d)
    got = _run_decode(ctx, e, q, hkv * n_rep, d, use_ring=False)
    ref = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], np.zeros(2, np.int64),
                                s, c, sk, hkv)
    assert allclose_report(got, ref)[0]


def test_decode_main_many_chunk_slots():
    """max_ctx far above the contexts: over 128 split-K chunk slots (the merge's general path) and a
    grid large enough for the separate query-fragment kernel."""
    d, hkv, n_rep, seed = 128, 1, 4, 91
    ctx, c, s, sk = make_ctx(tq, True, d, hkv * n_rep, hkv, seed)
    e = build_main_cache(seed, d, hkv, [2000, 700], c, s, sk)
    e["max_ctx"] = 320000
    q = synth.queries(seed, 2, hkv * n_rep, d)
    got = _run_decode(ctx, e, q, hkv * n_rep, d)
    ref = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], s, c, sk, hkv)
    ok, maxerr, nbad = allclose_report(got, ref)
    assert ok, f"max abs err {maxerr}, {nbad} elements outside 2e-3 + 1e-3|ref|"


def test_decode_empty_sequence_gives_zeros():
    d, hkv, seed = 128, 2, 5
    ctx, c, s, sk = make_ctx(tq, True, d, 4, hkv, seed)
    e = build_main_cache(seed, d, hkv, [0, 40], c, s, sk)
    q = synth.queries(seed, 2, 4, d)
    got = _run_decode(ctx, e, q, 4, d)
    assert np.all(got[0] == 0)
    ref = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], s, c, sk, hkv)
    assert allclose_report(got[1:], ref[1:])[0]


@pytest.mark.parametrize("d,n_rep", [(64, 1), (128, 1), (256, 1), (512, 1), (128, 2), (128, 8)])
def test_decode_alt_parity(d, n_rep):
    seed, hkv = 90 + d + n_rep, 2
    hq = hkv * n_rep
    ctx, c3, s, _ = make_ctx(tq, False, d, hq, hkv, seed)
    e = build_alt_cache(seed, d, hkv, [544, 96], c3, s)
    q = synth.queries(seed, 2, hq, d)
    out = torch.empty((2, hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(2, e["max_ctx"]), dtype=torch.uint8, device="cuda")
    ctx.decode_attention(to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), None, None, None,
                         e["max_ctx"], out, ws)
    got = out.cpu().numpy()
    assert ctx.device_errors() == 0
    ref = attention.decode_alt(q, e["pool"], e["bt"], e["n_c"], None, None, None, s, c3, hkv)
    ok, maxerr, nbad = allclose_report(got, ref)
    assert ok, f"max abs err {maxerr}, {nbad} bad"


# ====================================================================== append / ring
def test_append_ring_and_flush_on_overflow():
    d, hkv, seed, steps = 128, 2, 11, 260
    bsz = 2
    ctx, c, s, sk = make_ctx(tq, True, d, hkv * 2, hkv, seed)
    k, v = synth.kv_main(seed, bsz, hkv, steps, d)
    max_blocks = 20
    bt = synth.block_table(seed, bsz, max_blocks, True)
    pool_g = torch.zeros((bsz * max_blocks, hkv, layout.main_tile_bytes(d)), dtype=torch.uint8, device="cuda")
    ring_k = torch.zeros((bsz, hkv, 128, d), dtype=torch.float16, device="cuda")
    ring_v = torch.zeros_like(ring_k)
    kd, vd, btd = to_dev(k), to_dev(v), to_dev(bt)
    # sequence 1 starts 3 tokens behind sequence 0
    for step in range(steps):
        pos = np.array([step, max(step - 3, 0)], np.int32)
        kn = torch.stack([kd[0, :, step], kd[1, :, pos[1]]]).contiguous()
        vn = torch.stack([vd[0, :, step], vd[1, :, pos[1]]]).contiguous()
        if step < 3:  # sequence 1 idles: re-append its token 0 at position 0
            pass
        ctx.append_token(kn, vn, to_dev(pos), ring_k, ring_v, btd, pool_g)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    # sequence 0: 260 tokens -> 256 compressed, ring slots 0..3 hold tokens 256..259
    pool_o = np.zeros(pool_g.shape, np.uint8)
    enc = cache.encode_main_range(pool_o, bt[0:1], 0, k[0:1, :, :256], v[0:1, :, :256], s, c, sk)
    pg = pool_g.cpu().numpy()
    blocks = bt[0, :16]
    fo, fg = main_fields(pool_o[blocks], d), main_fields(pg[blocks], d)
    assert np.array_equal(fg["v_bytes"], fo["v_bytes"])
    yy = enc["y"][0].reshape(hkv, 16, 16, d).transpose(1, 0, 2, 3)
    assert not ((fg["idx"] != fo["idx"]) & ~near_boundary(yy, c)).any()
    rk = ring_k.cpu().numpy()
    assert np.array_equal(rk[0, :, :4], k[0, :, 256:260])
    # sequence 1 reached position 256: 256 tokens compressed (flush at 128 and 256), slot 0 = token 256
    assert np.array_equal(rk[1, :, 0], k[1, :, 256])
    assert np.array_equal(rk[1, :, 1:127], k[1, :, 129:255])


# ====================================================================== pack / errors
@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_device_pack_unpack_matches_oracle(bits):
    for n in (1, 31, 1000, 4097):
        codes = synth.random_codes(n * bits, n, bits)
        dev = tq.tq_pack(to_dev(codes), bits)
        got = dev.cpu().numpy()
        assert np.array_equal(got, layout.pack_bits(codes, bits))
        back = tq.tq_unpack(to_dev(layout.pack_bits(codes, bits)), n, bits).cpu().numpy()
        assert np.array_equal(back, codes)


def test_invalid_device_values_are_flagged_not_faulted():
    d, hkv, seed = 128, 2, 13
    ctx, c, s, sk = make_ctx(tq, True, d, 4, hkv, seed)
    e = build_main_cache(seed, d, hkv, [300, 200], c, s, sk)
    bt = e["bt"].copy()
    bt[0, 3] = 10_000_000  # block id beyond the pool
    e2 = dict(e, bt=bt)
    q = synth.queries(seed, 2, 4, d)
    out = torch.empty((2, 4, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(2, e["max_ctx"]), dtype=torch.uint8, device="cuda")
    n_b = e["n_b"].copy()
    n_b[1] = 500  # ring count beyond capacity
    ctx.decode_attention(to_dev(q), to_dev(e2["pool"]), to_dev(bt), to_dev(e["n_c"]), to_dev(e["ring_k"]),
                         to_dev(e["ring_v"]), to_dev(n_b), e["max_ctx"], out, ws)
    flags = ctx.device_errors()
    assert flags & tq.binding.TQ_DEVERR_BLOCK_ID and flags & tq.binding.TQ_DEVERR_RING
    assert np.all(np.isfinite(out.cpu().numpy()))
    # host-side checks: workspace too small, misaligned max_ctx
    with pytest.raises(tq.TQError) as err:
        ctx.decode_attention(to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), None, None, None,
                             e["max_ctx"], out, ws[:16])
    assert err.value.status == tq.binding.TQ_ERR_WORKSPACE
