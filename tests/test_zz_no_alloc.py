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
import numpy as np
import pytest
import torch

import synth
from gpu_cases import allclose_report, build_main_cache, make_ctx, to_dev

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


def test_static_entry_point_matches_workspace_entry_point_twice(tq):
    d, hkv, n_rep = 128, 4, 7
    hq = hkv * n_rep
    ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, 21)
    for call, (seed, lengths) in enumerate([(21, [3000, 130, 1]), (22, [700, 2049, 64, 5000])]):
        e = build_main_cache(seed, d, hkv, lengths, c, s, sk)
        assert ctx.workspace_size(len(lengths), e["max_ctx"]) <= STATIC_BYTES
        q = synth.queries(seed, len(lengths), hq, d)
        got, ref = _both(ctx, e, q, hq, d)
        ok, maxerr, nbad = allclose_report(got, ref)
        assert ok, f"call {call}: max abs err {maxerr}, {nbad} bad"
        assert np.all(np.isfinite(got))


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
