"""4-bit value codes in the main layout (turboquant vLLM guide, --value-bits 4) on the GPU.

The same parity bar as the 2-bit default: value planes bit-exact against the oracle's encoder,
key fields away from decision boundaries, decode within 2e-3 + 1e-3 |ref|, dequantised history
within half an fp16 step. d = 128 runs the tensor-core decoder, the other head dims the CUDA-core
one.
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


def test_record_size():
    ctx, *_ = make_ctx(tq, True, 128, 4, 4, 0, value_bits=4)
    assert ctx.bytes_per_token_head == 132 and ctx.page_bytes == layout.main_tile_bytes(128, 4)


@pytest.mark.parametrize("d", [128, 64, 512])
def test_encode_parity(d):
    n_tok = 256 if d <= 128 else 128
    starts = [0, 64]
    ctx, pool_o, pool_g, encs, bt, c = _encode_main_both(d, 2, n_tok, starts, seed=40 + d, value_bits=4)
    _compare_main(pool_o, pool_g, encs, bt, starts, n_tok, d, c)


@pytest.mark.parametrize("d,hkv,n_rep,lengths", [
    (128, 2, 4, [1500, 129, 16]),   # tensor-core decoder, ragged, ring-only row
    (128, 2, 7, [700]),
    (64, 2, 2, [900]),              # CUDA-core decoder
    (256, 1, 3, [640]),
    (512, 1, 8, [300]),
])
def test_decode_parity(d, hkv, n_rep, lengths):
    seed = 50 + d + n_rep
    hq = hkv * n_rep
    ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, seed, value_bits=4)
    e = build_main_cache(seed, d, hkv, lengths, c, s, sk, value_bits=4)
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


def test_append_flush_writes_4bit_pages():
    d, hkv, seed, steps = 128, 2, 13, 130
    ctx, c, s, sk = make_ctx(tq, True, d, hkv, hkv, seed, value_bits=4)
    k, v = synth.kv_main(seed, 1, hkv, steps, d)
    bt = synth.block_table(seed, 1, 10, True)
    pool_g = torch.zeros((10, hkv, layout.main_tile_bytes(d, 4)), dtype=torch.uint8, device="cuda")
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


@pytest.mark.parametrize("d", [128, 256])
def test_dequantize(d):
    seed, hkv = 60 + d, 2
    ctx, c, s, sk = make_ctx(tq, True, d, hkv, hkv, seed, value_bits=4)
    e = build_main_cache(seed, d, hkv, [400, 200], c, s, sk, value_bits=4)
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
