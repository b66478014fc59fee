"""Host-side checks of libtq (no GPU): exports, setup tables, host packing, argument validation."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import synth
from conftest import ROOT, golden
from oracle import codebook, layout, rng

from kv_cache_quantization_tq_gb300.build import build

build()
from kv_cache_quantization_tq_gb300 import binding as B  # noqa: E402


def _header_functions():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_function_is_exported_and_bound():
    names = _header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(B.lib, n), n
    assert sorted(B.EXPORTED) == names


def test_product_code_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "kv_cache_quantization_tq_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", text, re.M), f
                assert "oracle/" not in text, f


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_host_codebook_matches_oracle(d, bits):
    c, b = B.tq_lloyd_max(d, bits)
    co, bo = codebook.lloyd_max(d, bits)
    assert np.max(np.abs(c - co)) < 1e-9
    assert np.max(np.abs(b - bo)) < 1e-9
    assert np.array_equal(c, -c[::-1])


@pytest.mark.parametrize("d,bits", [(64, 5), (128, 6), (512, 7), (64, 8), (512, 8)])
def test_host_large_codebook_matches_oracle(d, bits):
    # 32..256 levels (q5_0 .. q8_0 values): both sides solve the fixed point by Newton's method,
    # the host with its own quadrature.  The host codebook satisfies the oracle's centroid
    # conditions to 1e-10 (scaled by sqrt(d)); at 256 levels the fixed point is weakly determined
    # (Lloyd's map contracts by 1 - O(1/K^2)), so that residual allows ~1e-9 between solutions.
    c, b = B.tq_lloyd_max(d, bits)
    co, bo = codebook.lloyd_max(d, bits)
    t, _, _ = codebook._cell_means(c, d)
    assert np.max(np.abs(t - c)) * np.sqrt(d) < 1e-10
    assert np.max(np.abs(c - co)) * np.sqrt(d) < 1e-8
    assert np.max(np.abs(b - bo)) * np.sqrt(d) < 1e-8
    assert np.array_equal(c, -c[::-1]) and np.all(np.diff(c) > 0)
    with pytest.raises(B.TQError):
        B.tq_lloyd_max(d, 9)


@pytest.mark.parametrize("seed", [0, 1, 12345, 2**63 + 7])
def test_host_tables_match_oracle_generator(seed):
    d = 128
    s, sk = B.tq_generate_tables(seed, d, d)
    assert np.array_equal(s, rng.signs(seed, d).astype(np.float32))
    ref = rng.gaussian_matrix(seed, d, d)
    ulp = np.spacing(np.abs(ref).astype(np.float32))
    assert np.all(np.abs(sk - ref) <= ulp)


@pytest.mark.parametrize("bits", list(range(1, 9)))
def test_host_pack_matches_oracle(bits):
    for n in (1, 5, 64, 333):
        codes = synth.random_codes(n + bits, n, bits)
        got = B.tq_pack_host(codes, bits)
        assert np.array_equal(got, layout.pack_bits(codes, bits))
        assert np.array_equal(B.tq_unpack_host(got, n, bits), codes)


def test_host_pack_golden_examples():
    for case in golden("pack_examples.json")["cases"]:
        got = B.tq_pack_host(np.array(case["codes"], np.uint8), case["bits"])
        assert got.tobytes().hex() == case["bytes_hex"]


def test_host_pack_rejects_out_of_range_codes():
    with pytest.raises(B.TQError):
        B.tq_pack_host(np.array([4], np.uint8), 2)


def test_config_validation():
    B.tq_config_init(B.TQ_LAYOUT_MAIN, 128, 28, 4)
    B.tq_config_init(B.TQ_LAYOUT_ALT, 512, 8, 8)
    B.tq_config_init(B.TQ_LAYOUT_MAIN, 128, 64, 4)  # n_rep 16 = 2 groups of 8
    with pytest.raises(B.TQError) as e:
        B.tq_config_init(B.TQ_LAYOUT_MAIN, 96, 16, 4)
    assert e.value.status == B.TQ_ERR_UNSUPPORTED
    with pytest.raises(B.TQError) as e:
        B.tq_config_init(B.TQ_LAYOUT_MAIN, 128, 10, 4)
    assert e.value.status == B.TQ_ERR_INVALID_ARG
    with pytest.raises(B.TQError) as e:
        B.tq_config_init(B.TQ_LAYOUT_MAIN, 128, 36, 4)  # n_rep 9 cannot split evenly
    assert e.value.status == B.TQ_ERR_UNSUPPORTED


def _cfg(lay, d, kb, vb, hq=8, hkv=4):
    cfg = B.tq_config_init(lay, d, hq, hkv)
    cfg.key_bits, cfg.value_bits = kb, vb
    return cfg


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_config_check_record_bytes_match_the_oracle_layouts(d):
    # every supported width: the C++ record size equals the oracle's tile size / 16
    for kb in (2, 3, 4):
        for vb in (2, 4):
            got = B.tq_config_check(_cfg(B.TQ_LAYOUT_MAIN, d, kb, vb))
            assert got == layout.main_bytes_per_token_head(d, vb, kb), (kb, vb)
    for kb in (2, 4, 5, 8, 16):
        for vb in (2, 3, 4, 5, 6, 7, 8):  # q2_0 .. q8_0 values
            got = B.tq_config_check(_cfg(B.TQ_LAYOUT_ALT, d, kb, vb))
            assert got == layout.alt_bytes_per_token_head(d, vb, kb), (kb, vb)
    assert B.tq_config_check(B.tq_config_init(B.TQ_LAYOUT_MAIN, d, 16, 4)) == 0.75 * d + 4
    assert B.tq_config_check(B.tq_config_init(B.TQ_LAYOUT_ALT, d, 8, 8)) == 1.5 * d + 2


def test_config_check_rejects_unsupported_widths():
    bad = [(B.TQ_LAYOUT_MAIN, 5, 2), (B.TQ_LAYOUT_MAIN, 1, 2), (B.TQ_LAYOUT_MAIN, 3, 3), (B.TQ_LAYOUT_MAIN, 3, 8),
           (B.TQ_LAYOUT_ALT, 3, 3), (B.TQ_LAYOUT_ALT, 6, 3), (B.TQ_LAYOUT_ALT, 7, 3), (B.TQ_LAYOUT_ALT, 12, 3),
           (B.TQ_LAYOUT_ALT, 8, 1), (B.TQ_LAYOUT_ALT, 8, 9), (B.TQ_LAYOUT_ALT, 16, 9)]
    for lay, kb, vb in bad:
        with pytest.raises(B.TQError) as e:
            B.tq_config_check(_cfg(lay, 128, kb, vb))
        assert e.value.status == B.TQ_ERR_UNSUPPORTED, (lay, kb, vb)
    cfg = _cfg(B.TQ_LAYOUT_MAIN, 128, 3, 2)
    cfg.qjl_m = 64  # the sketch is square
    with pytest.raises(B.TQError) as e:
        B.tq_config_check(cfg)
    assert e.value.status == B.TQ_ERR_UNSUPPORTED
    cfg = _cfg(B.TQ_LAYOUT_MAIN, 128, 3, 2)
    cfg.page_size = 32
    with pytest.raises(B.TQError) as e:
        B.tq_config_check(cfg)
    assert e.value.status == B.TQ_ERR_UNSUPPORTED
    assert B.lib.tq_config_check(None, None) == B.TQ_ERR_INVALID_ARG


def test_null_context_calls_are_rejected_without_cuda():
    lib = B.lib
    assert lib.tq_encode_flush(None, None, None, 1, 16, 16, None, None, 1, None, 1, None) == B.TQ_ERR_INVALID_ARG
    assert lib.tq_decode_attention(None, None, 1, None, 0, None, 0, None, None, None, None, 0, None, None, 0,
                                   None) == B.TQ_ERR_INVALID_ARG
    assert lib.tq_append_token(None, None, None, None, 1, None, None, None, 0, None, 0, None) == B.TQ_ERR_INVALID_ARG
    assert lib.tq_pack(None, 10, 9, None, None) == B.TQ_ERR_INVALID_ARG
    assert lib.tq_bytes_per_token_head(None) == 0
    assert lib.tq_launch_count(None) == 0
    assert lib.tq_status_string(B.TQ_ERR_WORKSPACE).startswith(b"TQ_ERR_WORKSPACE")
    assert lib.tq_workspace_size(None, 1, 16, C.byref(C.c_size_t())) == B.TQ_ERR_INVALID_ARG


def test_prefill_materialisation_rule():
    """vllm-metal TurboQuant guide, advanced settings: materialise when the history holds >= 8192
    tokens and the prefill chunk reaches 64 query tokens at head_dim 128, max(128, head_dim / 2)
    otherwise, within the MiB cap (0 switches materialisation off); decode steps never."""
    f = B.tq_should_materialize
    assert f(8192, 64, 128, 8) and not f(8191, 64, 128, 8) and not f(8192, 63, 128, 8)
    assert not f(100000, 1, 128, 8)                       # a decode step
    assert f(8192, 128, 64, 8) and not f(8192, 127, 64, 8)  # max(128, 32) = 128
    assert f(8192, 128, 256, 8) and not f(8192, 127, 256, 8)  # max(128, 128) = 128
    assert f(8192, 256, 512, 8) and not f(8192, 255, 512, 8)  # max(128, 256) = 256
    # dense K + V of 8192 tokens x 8 heads x 128 dims x 2 B = 32 MiB
    assert f(8192, 64, 128, 8, 32) and not f(8192, 64, 128, 8, 31)
    assert not f(8192, 64, 128, 8, 0) and f(8192, 64, 128, 8, -1)
    with pytest.raises(ValueError):
        f(-1, 64, 128, 8)


def test_int2_key_format_is_accepted_only_for_alternate_2_bit_keys():
    cfg = B.tq_config_init(B.TQ_LAYOUT_ALT, 128, 8, 8, 0)
    cfg.key_bits, cfg.key_format = 2, B.TQ_KEY_SIGNED
    assert B.tq_config_check(cfg) == 2 * 128 // 8 + 4 * 4 + 3 * 128 // 8 + 2  # the bytes of uint2
    cfg.key_bits = 8
    with pytest.raises(B.TQError):
        B.tq_config_check(cfg)
    main = B.tq_config_init(B.TQ_LAYOUT_MAIN, 128, 8, 8, 0)
    main.key_format = B.TQ_KEY_SIGNED
    with pytest.raises(B.TQError):
        B.tq_config_check(main)
