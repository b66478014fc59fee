"""Prefill materialisation on the GPU (tq_dequantize) against the oracle's dense history.

The oracle reconstructs in float64; the kernel computes in fp32 and stores fp16, so every element
must lie within half an fp16 step of the oracle's value (plus fp32 rounding), and values / ring rows
(sums of two fp16 numbers, or copies) must match the oracle rounded to fp16 almost everywhere.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_cases import build_alt_cache, build_main_cache, make_ctx, to_dev
from oracle import cache

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from kv_cache_quantization_tq_gb300.build import build

    build()
    import kv_cache_quantization_tq_gb300 as tq

SENTINEL = 0x7E00  # fp16 NaN bit pattern: rows that must stay untouched


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check_close(got16, ref64, what):
    """Half an fp16 step of the oracle's value, plus the fp32 arithmetic of a d-point butterfly
    (bounded relative to the row's norm, since every output mixes the whole row)."""
    got = got16.astype(np.float64)
    half_ulp = np.maximum(np.abs(ref64), 2.0 ** -14) * 2.0 ** -11
    row = np.linalg.norm(ref64, axis=-1, keepdims=True)
    err = np.abs(got - ref64)
    bad = err > half_ulp * 1.01 + 2e-6 * row + 1e-7
    assert not bad.any(), f"{what}: {bad.sum()} elements off, max err {err.max():.3g}"


def _outputs(bsz, hkv, max_tokens, d):
    k = torch.full((bsz, hkv, max_tokens, d), SENTINEL, dtype=torch.int16, device="cuda").view(torch.float16)
    v = torch.full((bsz, hkv, max_tokens, d), SENTINEL, dtype=torch.int16, device="cuda").view(torch.float16)
    return k, v


def _untouched(t, b, start):
    return bool((t[b, :, start:].view(torch.int16) == SENTINEL).all())


@pytest.mark.parametrize("d,hkv,lengths", [(128, 2, [300, 16, 1100, 129]), (64, 3, [250, 700]),
                                           (256, 2, [400, 130]), (512, 1, [300, 17])])
def test_main_layout_dense_history(d, hkv, lengths):
    seed = 21 + d
    ctx, c, s, sk = make_ctx(tq, True, d, 2 * hkv, hkv, seed)
    e = build_main_cache(seed, d, hkv, lengths, c, s, sk)
    bsz = len(lengths)
    max_tokens = ((max(lengths) + 15) // 16) * 16 + 32
    k_out, v_out = _outputs(bsz, hkv, max_tokens, d)
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), k_out, v_out,
                   to_dev(e["ring_k"]), to_dev(e["ring_v"]), to_dev(e["n_b"]))
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    kg, vg = k_out.cpu().numpy(), v_out.cpu().numpy()
    for b in range(bsz):
        nc, nb = int(e["n_c"][b]), int(e["n_b"][b])
        kr, vr = cache.materialize_main(e["pool"], e["bt"], b, nc, e["ring_k"], e["ring_v"], nb, s, c, sk, d)
        _check_close(kg[b, :, :nc + nb], kr, f"keys b={b}")
        _check_close(vg[b, :, :nc + nb], vr, f"values b={b}")
        # values and ring rows: one rounding of an exact fp32 result -> the oracle's fp16 almost everywhere
        assert np.mean(vg[b, :, :nc + nb] == vr.astype(np.float16)) > 0.999
        assert np.array_equal(kg[b, :, nc:nc + nb], e["ring_k"][b, :, :nb])
        assert _untouched(k_out, b, nc + nb) and _untouched(v_out, b, nc + nb)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_alt_layout_dense_history(d):
    seed, hkv = 31 + d, 2
    ctx, c3, s, _ = make_ctx(tq, False, d, hkv, hkv, seed)
    lengths = [320, 48, 160]
    e = build_alt_cache(seed, d, hkv, lengths, c3, s)
    bsz = len(lengths)
    max_tokens = 336
    k_out, v_out = _outputs(bsz, hkv, max_tokens, d)
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), k_out, v_out)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    kg, vg = k_out.cpu().numpy(), v_out.cpu().numpy()
    for b, L in enumerate(lengths):
        kr, vr = cache.materialize_alt(e["pool"], e["bt"], b, L, None, None, 0, s, c3, d)
        _check_close(kg[b, :, :L], kr, f"keys b={b}")
        _check_close(vg[b, :, :L], vr, f"values b={b}")
        assert np.mean(kg[b, :, :L] == kr.astype(np.float16)) > 0.999
        assert _untouched(k_out, b, L)


def test_bad_device_values_are_flagged_and_skipped():
    d, hkv = 128, 2
    ctx, c, s, sk = make_ctx(tq, True, d, hkv, hkv, 3)
    e = build_main_cache(3, d, hkv, [300, 300], c, s, sk)
    bt = e["bt"].copy()
    bt[0, 2] = 10 ** 6  # page 2 of sequence 0 points outside the pool
    n_c = e["n_c"].copy()
    k_out, v_out = _outputs(2, hkv, 320, d)
    ctx.dequantize(to_dev(e["pool"]), to_dev(bt), to_dev(n_c), k_out, v_out)
    torch.cuda.synchronize()
    assert ctx.device_errors() & tq.binding.TQ_DEVERR_BLOCK_ID
    assert bool((k_out[0, :, 32:48].view(torch.int16) == SENTINEL).all())  # the bad page is skipped
    kr, _ = cache.materialize_main(e["pool"], e["bt"], 1, int(n_c[1]), None, None, 0, s, c, sk, d)
    _check_close(k_out[1, :, :int(n_c[1])].cpu().numpy(), kr, "other sequence")
    n_c[1] = 40  # not page aligned
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(n_c), k_out, v_out)
    torch.cuda.synchronize()
    assert ctx.device_errors() & tq.binding.TQ_DEVERR_POSITION
    nb = np.array([0, 200], np.int32)  # more than the ring holds
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), k_out, v_out,
                   to_dev(e["ring_k"]), to_dev(e["ring_v"]), to_dev(nb))
    torch.cuda.synchronize()
    assert ctx.device_errors() & tq.binding.TQ_DEVERR_RING


def _check_close_bf16(got_bf16, ref64, what):
    """bf16 outputs: within half a bf16 step of the oracle's value (2^-8 relative at most), plus the
    fp32 arithmetic of the row's butterfly, as for fp16."""
    got = got_bf16.float().cpu().numpy().astype(np.float64)
    half_ulp = np.maximum(np.abs(ref64), 2.0 ** -126) * 2.0 ** -8
    row = np.linalg.norm(ref64, axis=-1, keepdims=True)
    err = np.abs(got - ref64)
    bad = err > half_ulp * 1.01 + 2e-6 * row + 1e-7
    assert not bad.any(), f"{what}: {bad.sum()} elements off, max err {err.max():.3g}"


@pytest.mark.parametrize("layout_main,d", [(True, 128), (True, 64), (False, 128), (False, 256)])
def test_dense_history_bf16(layout_main, d):
    """tq_dequantize_bf16 (the guide's FP16/BF16 materialisation): the same reconstruction rounded to
    bf16, ring rows converted from fp16."""
    seed, hkv = 41 + d, 2
    if layout_main:
        ctx, c, s, sk = make_ctx(tq, True, d, 2 * hkv, hkv, seed)
        lengths = [300, 1100, 16]
        e = build_main_cache(seed, d, hkv, lengths, c, s, sk)
    else:
        ctx, c, s, sk = make_ctx(tq, False, d, hkv, hkv, seed)
        lengths = [320, 48]
        e = build_alt_cache(seed, d, hkv, lengths, c, s)
    bsz = len(lengths)
    max_tokens = ((max(lengths) + 15) // 16) * 16 + 32
    k_out = torch.full((bsz, hkv, max_tokens, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    v_out = torch.full_like(k_out, float("nan"))
    ring = (to_dev(e["ring_k"]), to_dev(e["ring_v"]), to_dev(e["n_b"])) if layout_main else (None, None, None)
    ctx.dequantize(to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), k_out, v_out, *ring)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    for b in range(bsz):
        nc = int(e["n_c"][b])
        nb = int(e["n_b"][b]) if layout_main else 0
        if layout_main:
            kr, vr = cache.materialize_main(e["pool"], e["bt"], b, nc, e["ring_k"], e["ring_v"], nb, s, c, sk, d)
        else:
            kr, vr = cache.materialize_alt(e["pool"], e["bt"], b, nc, None, None, 0, s, c, d)
        _check_close_bf16(k_out[b, :, :nc + nb], kr, f"keys b={b}")
        _check_close_bf16(v_out[b, :, :nc + nb], vr, f"values b={b}")
        if nb:
            want = torch.from_numpy(e["ring_k"][b, :, :nb]).to(torch.bfloat16)
            assert torch.equal(k_out[b, :, nc:nc + nb].cpu(), want)
        assert bool(torch.isnan(k_out[b, :, nc + nb:].float()).all())  # rows past the history untouched
