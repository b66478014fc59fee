"""tq_decode_attention_static: decode attention for callers that cannot allocate.

Some callers cannot call cudaMalloc while they decode (a fixed memory budget
once serving starts, work being recorded into a CUDA graph, an allocator
owned by another runtime).  The static entry point keeps its split-K scratch
in a fixed 16 MiB device array inside the library instead of a caller
workspace.  These tests compare it, through the C ABI, with the ordinary
entry point on the same inputs, for two calls in a row with different
inputs, and check that a request larger than the array is refused.  This file
is collected last so that a failure here comes after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_cases import allclose_report, build_main_cache, make_ctx, to_dev
from oracle import attention

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_quantization_tq_gb300.build import build

    build()
    import kv_cache_quantization_tq_gb300 as mod

    return mod


def _both(ctx, e, q, hq, d):
    bsz = q.shape[0]
    args = (to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), to_dev(e["ring_k"]), to_dev(e["ring_v"]),
            to_dev(e["n_b"]))
    ref = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.workspace_size(bsz, e["max_ctx"]), dtype=torch.uint8, device="cuda")
    ctx.decode_attention(*args, e["max_ctx"], ref, ws)
    out = torch.full((bsz, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    ctx.decode_attention_static(*args, e["max_ctx"], out)
    torch.cuda.synchronize()
    assert ctx.device_errors() == 0
    return out.cpu().numpy(), ref.cpu().numpy()


@pytest.mark.parametrize("path", ["auto", "tcgen05"])
def test_static_entry_point_matches_workspace_entry_point_twice(tq, path):
    """Both entry points run the same kernels on the same plan, so their outputs are bit-identical;
    both also agree with the oracle to the decode tolerance."""
    d, hkv, n_rep = 128, 4, 7
    hq = hkv * n_rep
    ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, 21)
    ctx.set_decode_path(tq.TQ_DECODE_AUTO if path == "auto" else tq.TQ_DECODE_TCGEN05)
    for call, (seed, lengths) in enumerate([(21, [3000, 130, 1]), (22, [700, 2049, 64, 5000])]):
        e = build_main_cache(seed, d, hkv, lengths, c, s, sk)
        assert ctx.workspace_size(len(lengths), e["max_ctx"]) <= STATIC_BYTES
        q = synth.queries(seed, len(lengths), hq, d)
        got, ref = _both(ctx, e, q, hq, d)
        assert np.array_equal(got, ref), f"call {call}: outputs differ (max {np.max(np.abs(got - ref))})"
        orc = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], s, c, sk,
                                    hkv)
        ok, maxerr, nbad = allclose_report(got, orc)
        assert ok, f"call {call}: max abs err {maxerr} against the oracle, {nbad} bad"


def test_static_entry_point_checks_arguments_like_the_workspace_one(tq):
    """Identical status codes for identical bad arguments, before the scratch-size check; batch 0 is
    a no-op."""
    lib, vp = tq.binding.lib, ctypes.c_void_p
    ctx, c, s, sk = make_ctx(tq, True, 128, 8, 2, 25)
    dummy = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = vp(dummy.data_ptr())
    ws = vp(dummy.data_ptr())

    def both(q, batch, max_ctx):
        a = lib.tq_decode_attention(ctx.ptr, q, batch, p, 1, p, 1, p, None, None, None, max_ctx, p, ws,
                                    dummy.numel(), None)
        b = lib.tq_decode_attention_static(ctx.ptr, q, batch, p, 1, p, 1, p, None, None, None, max_ctx, p, None)
        return a, b

    assert both(p, 1, 100) == (tq.binding.TQ_ERR_INVALID_ARG,) * 2  # max_ctx not a multiple of 16
    assert both(None, 1, 64) == (tq.binding.TQ_ERR_INVALID_ARG,) * 2  # NULL q
    assert both(p, -1, 64) == (tq.binding.TQ_ERR_INVALID_ARG,) * 2
    assert both(p, 0, 64) == (tq.binding.TQ_OK,) * 2


def test_static_entry_point_refuses_oversized_requests(tq):
    ctx, c, s, sk = make_ctx(tq, True, 128, 40, 8, 23)
    big_ctx = 1 << 20  # far more split-K partials than the fixed array holds
    assert ctx.workspace_size(64, big_ctx) > STATIC_BYTES
    q = torch.zeros((64, 40, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros((64, 40, 128), dtype=torch.float32, device="cuda")
    bt = torch.zeros((64, 1), dtype=torch.int32, device="cuda")
    nc = torch.zeros(64, dtype=torch.int32, device="cuda")
    pool = torch.zeros((1, 8, ctx.page_bytes), dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.TQError) as err:
        ctx.decode_attention_static(q, pool, bt, nc, None, None, None, big_ctx, out)
    assert err.value.status == tq.binding.TQ_ERR_WORKSPACE
