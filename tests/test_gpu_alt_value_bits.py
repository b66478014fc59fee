"""Alternate layout with 2- or 4-bit value indices, and with 5-, 4- or 2-bit keys or fp16 keys, on
the GPU (vllm-metal TurboQuant guide, quantisation table: q2_0 / q4_0 values, q5_0 / q4_0 / uint2
keys; 8-bit keys with 4-bit values is its K8+V4 mix; fp16 keys are the V-only cache of the
"TurboQuant-MLX overview").

The same parity bar as the 3-bit default: key bytes bit-exact against the oracle's encoder, value
indices equal away from decision boundaries, value norms within one fp16 ulp, decode within
2e-3 + 1e-3 |ref| (the tensor-core warp-per-page decoder for 1, 2 or 4 heads per KV head, the
CUDA-core one for 8), dequantised history against the oracle's materialisation.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_cases import (allclose_report, alt_fields, build_alt_cache, make_ctx, near_boundary, oracle_tables, tile_index,
                       to_dev)
from oracle import attention, cache, layout
from test_gpu_dequant import _check_close, _outputs, _untouched

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from kv_cache_quantization_tq_gb300.build import build

    build()
    import kv_cache_quantization_tq_gb300 as tq


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("vb", [2, 4, 5, 8])
@pytest.mark.parametrize("d", [64, 512])
def test_record_size(d, vb):
    ctx, c, *_ = make_ctx(tq, False, d, 2, 2, 0, value_bits=vb)
    assert len(c) == 1 << vb
    assert ctx.bytes_per_token_head == d + 4 * (d // 32) + vb * d // 8 + 2
    assert ctx.page_bytes == layout.alt_tile_bytes(d, vb)


@pytest.mark.parametrize("vb", [2, 4, 5, 6, 7, 8])  # q2_0 .. q8_0 values (q3_0 is the default)
@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_encode_parity(d, vb):
    hkv, n_tok, starts, seed = 2, 96, [0, 32], 60 + d + vb
    ctx, c, s, _ = make_ctx(tq, False, d, hkv, hkv, seed, value_bits=vb)
    k, v = synth.kv_alt(seed, 2, hkv, n_tok, d)
    v[1, 1, 7] = 0  # zero value vector
    max_blocks = 10
    bt = synth.block_table(seed, 2, max_blocks, True)
    pool_o = np.zeros((2 * max_blocks, hkv, layout.alt_tile_bytes(d, vb)), np.uint8)
    encs = [cache.encode_alt_range(pool_o, bt[b:b + 1], starts[b], k[b:b + 1], v[b:b + 1], s, c) for b in range(2)]
    pool_g = torch.zeros(pool_o.shape, dtype=torch.uint8, device="cuda")
    ctx.encode_flush(to_dev(k), to_dev(v), to_dev(np.array(starts, np.int32)), to_dev(bt), pool_g)
    pool_g = pool_g.cpu().numpy()
    assert ctx.device_errors() == 0
    blocks = tile_index(bt, starts, n_tok)
    fo = alt_fields(pool_o[blocks], d)
    fg = alt_fields(pool_g[blocks], d)
    assert np.array_equal(fg["k_bytes"], fo["k_bytes"])  # affine int8 keys: bit-exact
    assert np.max(np.abs(fg["vn"].astype(np.int32) - fo["vn"].astype(np.int32))) <= 1
    y = np.stack([e["y"][0] for e in encs]).reshape(2, hkv, n_tok // 16, 16, d).transpose(0, 2, 1, 3, 4)
    near = near_boundary(y, c)
    assert not ((fg["vidx"] != fo["vidx"]) & ~near).any()
    if vb <= 4:
        assert fg["vidx"].max() == (1 << vb) - 1  # every level reachable: the stream width is used
    else:  # 32..256 levels: the top index bit is used (the outermost cells hold few samples)
        assert fg["vidx"].max() >= 1 << (vb - 1)


def _decode_case(d, n_rep, vb, kb, seed, lengths=(544, 96)):
    hkv = 2
    hq = hkv * n_rep
    ctx, c, s, _ = make_ctx(tq, False, d, hq, hkv, seed, value_bits=vb, key_bits=kb)
    e = build_alt_cache(seed, d, hkv, list(lengths), c, s, key_bits=kb)
    q = synth.queries(seed, len(lengths), hq, d)
    out = torch.empty((len(lengths), hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(len(lengths), e["max_ctx"]), dtype=torch.uint8, device="cuda")
    ctx.profile_begin()
    ctx.decode_attention(to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), None, None, None,
                         e["max_ctx"], out, ws)
    kernel = ctx.profile_end()["decode_kernel"]
    got = out.cpu().numpy()
    assert ctx.device_errors() == 0
    ref = attention.decode_alt(q, e["pool"], e["bt"], e["n_c"], None, None, None, s, c, hkv)
    ok, maxerr, nbad = allclose_report(got, ref)
    assert ok, f"max abs err {maxerr}, {nbad} bad"
    return kernel


@pytest.mark.parametrize("vb", [2, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("d,n_rep", [(64, 1), (128, 2), (128, 4), (256, 1), (512, 1), (128, 8)])
def test_decode_parity(d, n_rep, vb):
    kernel = _decode_case(d, n_rep, vb, 8, 70 + d + n_rep + vb)
    # up to 4 query heads per KV head (8-bit keys): the warp-per-page tensor-core decoder at every width
    assert kernel == ("decode_alt_v2_kernel" if n_rep <= 4 else "decode_alt_kernel"), kernel


@pytest.mark.parametrize("vb", [5, 8])
@pytest.mark.parametrize("d,n_rep", [(64, 2), (128, 1), (512, 1)])
def test_decode_parity_wide_values_fp16_keys(d, n_rep, vb):
    """q5_0 / q8_0 values beside fp16 keys (the V-only cache with wide values), ragged lengths with a
    partial last chunk."""
    kernel = _decode_case(d, n_rep, vb, 16, 170 + d + n_rep + vb, lengths=(1040, 16, 400))
    assert kernel == "decode_alt_v2_kernel", kernel


def test_decode_wide_values_low_bit_keys_use_the_cuda_core_decoder():
    """5- to 8-bit values with 2-, 4- or 5-bit keys: no tensor-core instance, same results."""
    kernel = _decode_case(128, 2, 6, 4, 311)
    assert kernel == "decode_alt_kernel", kernel


@pytest.mark.parametrize("vb", [2, 4, 6, 8])
@pytest.mark.parametrize("d", [64, 256])
def test_dense_history(d, vb):
    seed, hkv = 80 + d + vb, 2
    ctx, c, s, _ = make_ctx(tq, False, d, hkv, hkv, seed, value_bits=vb)
    lengths = [320, 48]
    e = build_alt_cache(seed, d, hkv, lengths, c, s)
    max_tokens = 336
    k_out, v_out = _outputs(len(lengths), hkv, max_tokens, d)
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), k_out, v_out)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    kg, vg = k_out.cpu().numpy(), v_out.cpu().numpy()
    for b, L in enumerate(lengths):
        kr, vr = cache.materialize_alt(e["pool"], e["bt"], b, L, None, None, 0, s, c, d)
        _check_close(kg[b, :, :L], kr, f"keys b={b}")
        _check_close(vg[b, :, :L], vr, f"values b={b}")
        assert _untouched(k_out, b, L)


# ---- keys below 8 bits (q5_0 / q4_0 / uint2: 31-, 15- or 3-step affine codes per block of 32, a
# dense kb-bit stream per token)
@pytest.mark.parametrize("kb", [5, 4, 2])
@pytest.mark.parametrize("vb", [3, 4])
@pytest.mark.parametrize("d", [64, 128, 512])
def test_encode_parity_low_bit_keys(d, vb, kb):
    hkv, n_tok, starts, seed = 2, 96, [0, 32], 90 + d + vb + 7 * kb
    ctx, c, s, _ = make_ctx(tq, False, d, hkv, hkv, seed, value_bits=vb, key_bits=kb)
    assert ctx.bytes_per_token_head == kb * d // 8 + 4 * (d // 32) + vb * d // 8 + 2
    assert ctx.page_bytes == layout.alt_tile_bytes(d, vb, kb)
    k, v = synth.kv_alt(seed, 2, hkv, n_tok, d)
    max_blocks = 10
    bt = synth.block_table(seed, 2, max_blocks, True)
    pool_o = np.zeros((2 * max_blocks, hkv, layout.alt_tile_bytes(d, vb, kb)), np.uint8)
    encs = [cache.encode_alt_range(pool_o, bt[b:b + 1], starts[b], k[b:b + 1], v[b:b + 1], s, c) for b in range(2)]
    pool_g = torch.zeros(pool_o.shape, dtype=torch.uint8, device="cuda")
    ctx.encode_flush(to_dev(k), to_dev(v), to_dev(np.array(starts, np.int32)), to_dev(bt), pool_g)
    pool_g = pool_g.cpu().numpy()
    assert ctx.device_errors() == 0
    blocks = tile_index(bt, starts, n_tok)
    fo = alt_fields(pool_o[blocks], d, kb)
    fg = alt_fields(pool_g[blocks], d, kb)
    assert np.array_equal(fg["k_bytes"], fo["k_bytes"])  # affine key codes and their scales: bit-exact
    assert np.max(np.abs(fg["vn"].astype(np.int32) - fo["vn"].astype(np.int32))) <= 1
    y = np.stack([e["y"][0] for e in encs]).reshape(2, hkv, n_tok // 16, 16, d).transpose(0, 2, 1, 3, 4)
    assert not ((fg["vidx"] != fo["vidx"]) & ~near_boundary(y, c)).any()
    kq = layout.unpack_alt_tiles(pool_g[blocks], d, vb)["kq"]
    assert kq.max() == (1 << kb) - 1  # the top code is reached: the stream width is used


@pytest.mark.parametrize("kb", [5, 4, 2, 16])
@pytest.mark.parametrize("d,n_rep", [(64, 1), (128, 2), (256, 1), (512, 1), (128, 4), (128, 8)])
def test_decode_parity_low_bit_keys(d, n_rep, kb):
    seed, hkv, vb = 100 + d + n_rep + 7 * kb, 2, 3
    hq = hkv * n_rep
    ctx, c, s, _ = make_ctx(tq, False, d, hq, hkv, seed, value_bits=vb, key_bits=kb)
    e = build_alt_cache(seed, d, hkv, [544, 96], c, s, key_bits=kb)
    q = synth.queries(seed, 2, hq, d)
    out = torch.empty((2, hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(2, e["max_ctx"]), dtype=torch.uint8, device="cuda")
    ctx.decode_attention(to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), None, None, None,
                         e["max_ctx"], out, ws)
    got = out.cpu().numpy()
    assert ctx.device_errors() == 0
    ref = attention.decode_alt(q, e["pool"], e["bt"], e["n_c"], None, None, None, s, c, hkv)
    ok, maxerr, nbad = allclose_report(got, ref)
    assert ok, f"max abs err {maxerr}, {nbad} bad"


@pytest.mark.parametrize("kb", [5, 4, 2, 16])
@pytest.mark.parametrize("d", [64, 256])
def test_dense_history_low_bit_keys(d, kb):
    seed, hkv, vb = 110 + d + 7 * kb, 2, 3
    ctx, c, s, _ = make_ctx(tq, False, d, hkv, hkv, seed, value_bits=vb, key_bits=kb)
    lengths = [320, 48]
    e = build_alt_cache(seed, d, hkv, lengths, c, s, key_bits=kb)
    max_tokens = 336
    k_out, v_out = _outputs(len(lengths), hkv, max_tokens, d)
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), k_out, v_out)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    kg, vg = k_out.cpu().numpy(), v_out.cpu().numpy()
    for b, L in enumerate(lengths):
        kr, vr = cache.materialize_alt(e["pool"], e["bt"], b, L, None, None, 0, s, c, d)
        _check_close(kg[b, :, :L], kr, f"keys b={b}")
        _check_close(vg[b, :, :L], vr, f"values b={b}")
        assert _untouched(k_out, b, L)


# ---- fp16 keys, quantised values only (the V-only cache)
@pytest.mark.parametrize("vb", [2, 3, 4])
@pytest.mark.parametrize("d", [64, 128, 512])
def test_encode_parity_fp16_keys(d, vb):
    hkv, n_tok, starts, seed = 2, 96, [0, 32], 120 + d + vb
    ctx, c, s, _ = make_ctx(tq, False, d, hkv, hkv, seed, value_bits=vb, key_bits=16)
    assert ctx.bytes_per_token_head == 2 * d + vb * d // 8 + 2
    assert ctx.page_bytes == layout.alt_tile_bytes(d, vb, 16)
    k, v = synth.kv_alt(seed, 2, hkv, n_tok, d)
    max_blocks = 10
    bt = synth.block_table(seed, 2, max_blocks, True)
    pool_o = np.zeros((2 * max_blocks, hkv, layout.alt_tile_bytes(d, vb, 16)), np.uint8)
    encs = [cache.encode_alt_range(pool_o, bt[b:b + 1], starts[b], k[b:b + 1], v[b:b + 1], s, c) for b in range(2)]
    pool_g = torch.zeros(pool_o.shape, dtype=torch.uint8, device="cuda")
    ctx.encode_flush(to_dev(k), to_dev(v), to_dev(np.array(starts, np.int32)), to_dev(bt), pool_g)
    pool_g = pool_g.cpu().numpy()
    assert ctx.device_errors() == 0
    blocks = tile_index(bt, starts, n_tok)
    fo = alt_fields(pool_o[blocks], d, 16)
    fg = alt_fields(pool_g[blocks], d, 16)
    assert np.array_equal(fg["k_bytes"], fo["k_bytes"])  # the fp16 keys, bit for bit
    k16 = layout.unpack_alt_tiles(pool_g[blocks], d, vb)["k16"]
    assert np.array_equal(k16[0, 0, 0].view(np.uint16), k[0, 0, :16].view(np.uint16))
    assert np.max(np.abs(fg["vn"].astype(np.int32) - fo["vn"].astype(np.int32))) <= 1
    y = np.stack([e["y"][0] for e in encs]).reshape(2, hkv, n_tok // 16, 16, d).transpose(0, 2, 1, 3, 4)
    assert not ((fg["vidx"] != fo["vidx"]) & ~near_boundary(y, c)).any()


# ---- int2 keys: signed symmetric mid-rise 2-bit codes (TQ_KEY_SIGNED), the vllm-metal int2 / q2_0 row
def _int2_ctx(d, hq, hkv, seed, vb):
    c32, signs, _ = oracle_tables(seed, d, False, 3, vb)
    ctx = tq.Context(tq.TQ_LAYOUT_ALT, d, hq, hkv, seed, centroids=c32, signs=signs, value_bits=vb, key_bits=2,
                     key_format=tq.TQ_KEY_SIGNED)
    return ctx, c32.astype(np.float64), signs.astype(np.float64)


@pytest.mark.parametrize("d,vb", [(128, 2), (64, 3), (512, 2)])
def test_int2_keys_encode_decode_dequantize(d, vb):
    hkv, n_tok, starts, seed = 2, 96, [0, 32], 130 + d + vb
    ctx, c, s = _int2_ctx(d, 2 * hkv, hkv, seed, vb)
    assert ctx.bytes_per_token_head == 2 * d // 8 + 4 * (d // 32) + vb * d // 8 + 2  # the bytes of uint2
    k, v = synth.kv_alt(seed, 2, hkv, n_tok, d)
    max_blocks = 10
    bt = synth.block_table(seed, 2, max_blocks, True)
    pool_o = np.zeros((2 * max_blocks, hkv, layout.alt_tile_bytes(d, vb, 2)), np.uint8)
    for b in range(2):
        cache.encode_alt_range(pool_o, bt[b:b + 1], starts[b], k[b:b + 1], v[b:b + 1], s, c, key_signed=True)
    pool_g = torch.zeros(pool_o.shape, dtype=torch.uint8, device="cuda")
    ctx.encode_flush(to_dev(k), to_dev(v), to_dev(np.array(starts, np.int32)), to_dev(bt), pool_g)
    pool_g = pool_g.cpu().numpy()
    assert ctx.device_errors() == 0
    blocks = tile_index(bt, starts, n_tok)
    fo, fg = alt_fields(pool_o[blocks], d, 2), alt_fields(pool_g[blocks], d, 2)
    assert np.array_equal(fg["k_bytes"], fo["k_bytes"])  # signed codes and their (s, mn): bit-exact
    # decode and dequantise an oracle-encoded int2 cache
    e = build_alt_cache(seed, d, hkv, [544, 96], c, s, key_bits=2, key_signed=True)
    q = synth.queries(seed, 2, 2 * hkv, d)
    out = torch.empty((2, 2 * hkv, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(2, e["max_ctx"]), dtype=torch.uint8, device="cuda")
    ctx.decode_attention(to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), None, None, None,
                         e["max_ctx"], out, ws)
    assert ctx.device_errors() == 0
    ref = attention.decode_alt(q, e["pool"], e["bt"], e["n_c"], None, None, None, s, c, hkv)
    ok, maxerr, nbad = allclose_report(out.cpu().numpy(), ref)
    assert ok, f"max abs err {maxerr}, {nbad} bad"
    k_out, v_out = _outputs(2, hkv, 560, d)
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), k_out, v_out)
    torch.cuda.synchronize()
    kg = k_out.cpu().numpy()
    for b, L in enumerate([544, 96]):
        kr, _ = cache.materialize_alt(e["pool"], e["bt"], b, L, None, None, 0, s, c, d)
        _check_close(kg[b, :, :L], kr, f"keys b={b}")
