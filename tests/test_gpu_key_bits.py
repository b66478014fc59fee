"""2- and 4-bit keys in the main layout (turboquant vLLM guide, --key-bits) on the GPU: a 1-bit
Lloyd-Max index (centroids +-E|x|) or a 3-bit one (8 centroids), each with the 1-bit QJL sketch,
and 2- or 4-bit values.

Same parity bar as the default layout; d = 128 runs the tensor-core decoder (two bit planes for
2-bit keys; for 4-bit keys the three index planes, their XOR and the QJL plane), other head dims
the CUDA-core one.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_cases import allclose_report, build_main_cache, make_ctx, main_fields, near_boundary, to_dev
from oracle import attention, cache, layout
from test_gpu_parity import _compare_main, _encode_main_both

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from kv_cache_quantization_tq_gb300.build import build

    build()
    import kv_cache_quantization_tq_gb300 as tq


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_record_size_4bit_keys():
    ctx, c, *_ = make_ctx(tq, True, 128, 4, 4, 0, key_bits=4)
    assert ctx.bytes_per_token_head == 116 and len(c) == 8
    lib_ctx = tq.Context(tq.TQ_LAYOUT_MAIN, 128, 4, 4, 0, key_bits=4)
    assert np.allclose(lib_ctx.get_tables()["centroids"], c, rtol=1e-6)


@pytest.mark.parametrize("kb", [2, 4])
def test_dequantize(kb):
    d, hkv, seed = 128, 2, 90 + kb
    ctx, c, s, sk = make_ctx(tq, True, d, hkv, hkv, seed, key_bits=kb)
    e = build_main_cache(seed, d, hkv, [400, 200], c, s, sk, key_bits=kb)
    k_out = torch.zeros((2, hkv, 416, d), dtype=torch.float16, device="cuda")
    v_out = torch.zeros_like(k_out)
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), k_out, v_out, to_dev(e["ring_k"]),
                   to_dev(e["ring_v"]), to_dev(e["n_b"]))
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    kg, vg = k_out.cpu().numpy().astype(np.float64), v_out.cpu().numpy().astype(np.float64)
    for b in range(2):
        nc, nb = int(e["n_c"][b]), int(e["n_b"][b])
        kr, vr = cache.materialize_main(e["pool"], e["bt"], b, nc, e["ring_k"], e["ring_v"], nb, s, c, sk, d)
        for got, ref in ((kg[b, :, :nc + nb], kr), (vg[b, :, :nc + nb], vr)):
            half_ulp = np.maximum(np.abs(ref), 2.0 ** -14) * 2.0 ** -11
            row = np.linalg.norm(ref, axis=-1, keepdims=True)
            assert np.all(np.abs(got - ref) <= half_ulp * 1.01 + 2e-6 * row + 1e-7)


def test_record_size_and_codebook():
    ctx, c, *_ = make_ctx(tq, True, 128, 4, 4, 0, key_bits=2)
    assert ctx.bytes_per_token_head == 84 and ctx.page_bytes == layout.main_tile_bytes(128, 2, 2)
    ctx2 = tq.Context(tq.TQ_LAYOUT_MAIN, 128, 4, 4, 0, key_bits=2, value_bits=4)  # library's own codebook
    assert ctx2.bytes_per_token_head == 116
    # the library's own 1-bit codebook: +-E|x| of a sphere coordinate, as the oracle's
    assert np.allclose(ctx2.get_tables()["centroids"], c, rtol=1e-6)


@pytest.mark.parametrize("d,vb,kb", [(128, 2, 2), (64, 4, 2), (512, 2, 2), (128, 2, 4), (256, 4, 4)])
def test_encode_parity(d, vb, kb):
    n_tok = 256 if d <= 128 else 128
    starts = [0, 32]
    ctx, pool_o, pool_g, encs, bt, c = _encode_main_both(d, 2, n_tok, starts, seed=70 + d, value_bits=vb, key_bits=kb)
    _compare_main(pool_o, pool_g, encs, bt, starts, n_tok, d, c)


@pytest.mark.parametrize("d,vb,kb,hkv,n_rep,lengths", [
    (128, 2, 2, 2, 4, [1500, 129, 16]),   # tensor-core decoder
    (128, 4, 2, 2, 7, [700]),
    (64, 2, 2, 2, 2, [900]),              # CUDA-core decoder
    (256, 4, 2, 1, 3, [640]),
    (128, 2, 4, 2, 4, [1500, 129, 16]),   # 4-bit keys: tensor-core
    (128, 4, 4, 1, 8, [900]),
    (64, 2, 4, 2, 2, [700]),              # 4-bit keys: CUDA-core
])
def test_decode_parity(d, vb, kb, hkv, n_rep, lengths):
    seed = 80 + d + n_rep + kb
    hq = hkv * n_rep
    ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, seed, value_bits=vb, key_bits=kb)
    e = build_main_cache(seed, d, hkv, lengths, c, s, sk, value_bits=vb, key_bits=kb)
    q = synth.queries(seed, len(lengths), hq, d)
    out = torch.empty((len(lengths), hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(len(lengths), e["max_ctx"]), dtype=torch.uint8, device="cuda")
    ctx.decode_attention(to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), to_dev(e["ring_k"]),
                         to_dev(e["ring_v"]), to_dev(e["n_b"]), e["max_ctx"], out, ws)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    ref = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], s, c, sk, hkv)
    ok, maxerr, nbad = allclose_report(out.cpu().numpy(), ref)
    assert ok, f"max abs err {maxerr}, {nbad} elements outside 2e-3 + 1e-3|ref|"


def test_append_flush_and_dequantize():
    d, hkv, seed, steps = 128, 2, 17, 130
    ctx, c, s, sk = make_ctx(tq, True, d, hkv, hkv, seed, key_bits=2)
    k, v = synth.kv_main(seed, 1, hkv, steps, d)
    bt = synth.block_table(seed, 1, 10, True)
    pool_g = torch.zeros((10, hkv, layout.main_tile_bytes(d, 2, 2)), dtype=torch.uint8, device="cuda")
    ring_k = torch.zeros((1, hkv, 128, d), dtype=torch.float16, device="cuda")
    ring_v = torch.zeros_like(ring_k)
    kd, vd, btd = to_dev(k), to_dev(v), to_dev(bt)
    for step in range(steps):
        ctx.append_token(kd[:, :, step].contiguous(), vd[:, :, step].contiguous(), to_dev(np.array([step], np.int32)),
                         ring_k, ring_v, btd, pool_g)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    pool_o = np.zeros(pool_g.shape, np.uint8)
    enc = cache.encode_main_range(pool_o, bt, 0, k[:, :, :128], v[:, :, :128], s, c, sk)
    blocks = bt[0, :8]
    fo, fg = main_fields(pool_o[blocks], d), main_fields(pool_g.cpu().numpy()[blocks], d)
    assert np.array_equal(fg["v_bytes"], fo["v_bytes"])
    yy = enc["y"][0].reshape(hkv, 8, 16, d).transpose(1, 0, 2, 3)
    assert not ((fg["idx"] != fo["idx"]) & ~near_boundary(yy, c)).any()
    # dense history from the oracle's pages (so no GPU encoding enters the reference)
    pool_d = to_dev(pool_o)
    k_out = torch.zeros((1, hkv, 144, d), dtype=torch.float16, device="cuda")
    v_out = torch.zeros_like(k_out)
    ctx.dequantize(pool_d, btd, to_dev(np.array([128], np.int32)), k_out, v_out, ring_k, ring_v,
                   to_dev(np.array([2], np.int32)))
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    kr, vr = cache.materialize_main(pool_o, bt, 0, 128, ring_k.cpu().numpy(), ring_v.cpu().numpy(), 2, s, c, sk, d)
    for got, ref in ((k_out[0, :, :130].cpu().numpy().astype(np.float64), kr),
                     (v_out[0, :, :130].cpu().numpy().astype(np.float64), vr)):
        half_ulp = np.maximum(np.abs(ref), 2.0 ** -14) * 2.0 ** -11
        row = np.linalg.norm(ref, axis=-1, keepdims=True)
        assert np.all(np.abs(got - ref) <= half_ulp * 1.01 + 2e-6 * row + 1e-7)
