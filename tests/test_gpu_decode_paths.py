"""Both main-layout decode designs against the CPU oracle, through the C ABI (GPU).

TQ_DECODE_MMA_SYNC scores and accumulates on mma.sync; TQ_DECODE_TCGEN05 scores on tcgen05 with
fp8 key bytes in tensor memory (3-bit keys, 2-bit values).  Each case runs both, on the same
oracle-encoded cache, to the decode tolerance 2e-3 + 1e-3 |ref|."""
import numpy as np
import pytest
import torch

import synth
from gpu_cases import allclose_report, build_main_cache, make_ctx, to_dev
from oracle import attention

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from kv_cache_quantization_tq_gb300.build import build

    build()
    import kv_cache_quantization_tq_gb300 as tq

    PATHS = [tq.TQ_DECODE_MMA_SYNC, tq.TQ_DECODE_TCGEN05]
else:  # collected on CPU-only hosts, deselected by -m "not gpu"
    tq = None
    PATHS = [1, 2]


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _decode(ctx, e, q, hq, d, max_ctx=None):
    bsz = q.shape[0]
    max_ctx = e["max_ctx"] if max_ctx is None else max_ctx
    out = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(ctx.workspace_size(bsz, max_ctx), 1), dtype=torch.uint8, device="cuda")
    ctx.decode_attention(to_dev(q), to_dev(e["pool"]), to_dev(e["bt"]), to_dev(e["n_c"]), to_dev(e["ring_k"]),
                         to_dev(e["ring_v"]), to_dev(e["n_b"]), max_ctx, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _case(path, hkv, n_rep, lengths, seed, v_scale=1.0, max_ctx=None):
    d, hq = 128, hkv * n_rep
    ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, seed)
    ctx.set_decode_path(path)
    e = build_main_cache(seed, d, hkv, lengths, c, s, sk, v_scale=v_scale)
    q = synth.queries(seed, len(lengths), hq, d)
    got = _decode(ctx, e, q, hq, d, max_ctx)
    assert ctx.device_errors() == 0
    ref = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], s, c, sk, hkv)
    return allclose_report(got, ref)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("hkv,n_rep,lengths", [
    (4, 4, [1024]),                    # single decode step geometry: 7 pages, one partial tile
    (2, 7, [1500, 300, 17, 128]),      # GQA 7, ragged, ring-only rows
    (2, 5, [2049, 129]),               # one-token rings
    (1, 16, [700]),                    # two head groups per KV head
    (3, 1, [333]),
    (2, 8, [9000, 4100]),              # several 8-page tiles and chunks, partial last tile
    (1, 6, [145]),                     # a single compressed page
])
def test_decode_paths_parity(path, hkv, n_rep, lengths):
    ok, maxerr, nbad = _case(path, hkv, n_rep, lengths, seed=31 * n_rep + hkv + len(lengths))
    assert ok, f"max abs err {maxerr}, {nbad} elements outside 2e-3 + 1e-3|ref|"


@pytest.mark.parametrize("path", PATHS)
def test_decode_paths_large_values(path):
    """Value groups with ranges of ~1e3..1e4 (values x 200): their fp16 scales times softmax weights
    of up to 2^8 must stay inside the fp16 operands of the value product."""
    ok, maxerr, nbad = _case(path, 2, 4, [3000, 640], seed=5, v_scale=200.0)
    assert ok, f"max abs err {maxerr}, {nbad} elements outside 2e-3 + 1e-3|ref|"


@pytest.mark.parametrize("path", PATHS)
def test_decode_paths_many_chunks(path):
    """max_ctx far above the contexts: many split-K chunk slots, most of them empty."""
    ok, maxerr, nbad = _case(path, 1, 4, [2000, 700], seed=91, max_ctx=320000)
    assert ok, f"max abs err {maxerr}, {nbad} elements outside 2e-3 + 1e-3|ref|"


def test_tcgen05_bad_block_id_is_flagged():
    d, hkv, n_rep, seed = 128, 2, 4, 13
    ctx, c, s, sk = make_ctx(tq, True, d, hkv * n_rep, hkv, seed)
    ctx.set_decode_path(tq.TQ_DECODE_TCGEN05)
    e = build_main_cache(seed, d, hkv, [1200, 800], c, s, sk)
    e["bt"] = e["bt"].copy()
    e["bt"][0, 5] = e["pool"].shape[0] + 7  # outside the pool
    q = synth.queries(seed, 2, hkv * n_rep, d)
    _decode(ctx, e, q, hkv * n_rep, d)
    assert ctx.device_errors() & tq.binding.TQ_DEVERR_BLOCK_ID


def test_decode_path_rejects_unknown_value():
    d, seed = 128, 3
    ctx, c, s, sk = make_ctx(tq, True, d, 4, 1, seed)
    with pytest.raises(tq.TQError):
        ctx.set_decode_path(7)


@pytest.mark.parametrize("path", PATHS)
def test_consecutive_calls_on_one_context(path):
    """Calls of different batch sizes and split-K plans back to back on one context (a one-wave
    plan, a single sequence, a four-sequence batch, a plan sized for 128K tokens, then the first
    call again), each checked against the oracle: no state of one call may leak into the next."""
    d, hkv, n_rep, seed = 128, 2, 4, 61
    hq = hkv * n_rep
    ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, seed)
    ctx.set_decode_path(path)
    cases = [([2000, 700, 5], None), ([300], None), ([4096, 4096, 1200, 33], None), ([1500, 20], 1 << 17),
             ([2000, 700, 5], None)]
    for k, (lengths, max_ctx) in enumerate(cases):
        e = build_main_cache(seed + k, d, hkv, lengths, c, s, sk)
        q = synth.queries(seed + k, len(lengths), hq, d)
        got = _decode(ctx, e, q, hq, d, max_ctx)
        assert ctx.device_errors() == 0
        ref = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], s, c, sk,
                                    hkv)
        ok, maxerr, nbad = allclose_report(got, ref)
        assert ok, f"call {k} ({lengths}): max abs err {maxerr}, {nbad} bad"


@pytest.mark.parametrize("path", PATHS)
def test_repeated_decodes_are_bit_identical(path):
    """Each decoder's arithmetic order is fixed (per-CTA combine order, lazy reference updates,
    merge order), so the same inputs give the same bits on every call; a race between warp roles
    or CTAs would show as a difference.  Twenty calls per shape, the first also against the
    oracle."""
    d = 128
    for k, (hkv, n_rep, lengths) in enumerate([(2, 7, [5000, 130, 2049]), (4, 4, [777]), (1, 16, [3000, 1])]):
        hq = hkv * n_rep
        seed = 71 + k
        ctx, c, s, sk = make_ctx(tq, True, d, hq, hkv, seed)
        ctx.set_decode_path(path)
        e = build_main_cache(seed, d, hkv, lengths, c, s, sk)
        q = synth.queries(seed, len(lengths), hq, d)
        first = _decode(ctx, e, q, hq, d)
        assert ctx.device_errors() == 0
        ref = attention.decode_main(q, e["pool"], e["bt"], e["n_c"], e["ring_k"], e["ring_v"], e["n_b"], s, c, sk,
                                    hkv)
        ok, maxerr, nbad = allclose_report(first, ref)
        assert ok, f"shape {k}: max abs err {maxerr}, {nbad} bad"
        for it in range(19):
            again = _decode(ctx, e, q, hq, d)
            assert np.array_equal(again, first), f"shape {k}, call {it + 2}: output differs from the first call"
        assert ctx.device_errors() == 0
