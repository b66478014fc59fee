"""Pins for the oracle's bit packing, tile layouts and byte counts."""
import numpy as np
import pytest

import synth
from oracle import cache, layout
from conftest import golden


def _pack_bigint(codes, bits):
    """Brute force: the stream as one little-endian integer sum(code_i << bits*i)."""
    v = 0
    for i, c in enumerate(codes):
        v |= int(c) << (bits * i)
    n = (len(codes) * bits + 7) // 8
    return np.frombuffer(v.to_bytes(n, "little"), dtype=np.uint8)


def test_hand_worked_examples():
    for case in golden("pack_examples.json")["cases"]:
        got = layout.pack_bits(np.array(case["codes"], np.uint8), case["bits"])
        assert got.tobytes().hex() == case["bytes_hex"], case
        back = layout.unpack_bits(got, len(case["codes"]), case["bits"])
        assert back.tolist() == case["codes"]


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n", [1, 7, 32, 100, 129])
def test_round_trip_and_bigint(bits, n):
    codes = synth.random_codes(n * 10 + bits, n, bits)
    packed = layout.pack_bits(codes, bits)
    assert packed.size == layout.packed_size(n, bits)
    assert np.array_equal(packed, _pack_bigint(codes, bits))
    assert np.array_equal(layout.unpack_bits(packed, n, bits), codes)
    rows = np.stack([codes] * 3)
    if (n * bits) % 8 == 0:
        pr = layout.pack_rows(rows, bits)
        assert np.array_equal(pr[1], packed)
        assert np.array_equal(layout.unpack_rows(pr, n, bits), rows)


def test_three_bit_32_values_fill_12_bytes():
    assert layout.packed_size(32, 3) == 12
    assert layout.pack_bits(np.full(32, 7, np.uint8), 3).tolist() == [255] * 12


def test_plane_words_brute_force():
    bits = synth.random_codes(1, 3 * 128, 1).reshape(3, 128)
    words = layout.bits_to_plane_words(bits)
    for r in range(3):
        for w in range(4):
            want = 0
            for j in range(16):
                for e in range(2):
                    want |= int(bits[r, 32 * w + 2 * j + e]) << (16 * e + j)
            assert int(words[r, w]) == want
    assert np.array_equal(layout.plane_words_to_bits(words), bits)


def test_vq_words_brute_force():
    codes = synth.random_codes(2, 16 * 64, 2).reshape(16, 64)
    words = layout.codes_to_vq_words(codes)
    for i in range(64):
        want = 0
        for t in range(16):
            j, e = divmod(t, 2)
            want |= int(codes[t, i]) << (16 * e + 2 * j)
        assert int(words[i]) == want
    assert np.array_equal(layout.vq_words_to_codes(words), codes)


def test_vq_words_4bit_brute_force_and_hand_worked():
    # word w of a dimension holds tokens 8w + 2j + e at bit 16e + 4j; all w = 0 words first
    codes = synth.random_codes(3, 16 * 32, 4).reshape(16, 32)
    words = layout.codes_to_vq_words(codes, 4)
    assert words.shape == (64,)
    for i in range(32):
        for w in range(2):
            want = 0
            for t in range(8):
                j, e = divmod(t, 2)
                want |= int(codes[8 * w + t, i]) << (16 * e + 4 * j)
            assert int(words[w * 32 + i]) == want
    assert np.array_equal(layout.vq_words_to_codes(words, 4), codes)
    # token t carries code t in every dimension
    ramp = np.repeat(np.arange(16, dtype=np.uint8)[:, None], 4, axis=1)
    w = layout.codes_to_vq_words(ramp, 4)
    assert int(w[0]) == 0x75316420 and int(w[4]) == 0xFDB9ECA8


@pytest.mark.parametrize("d", [64, 256])
def test_main_tile_round_trip_4bit_values(d):
    g = np.random.default_rng(d + 1)
    f = {
        "idx": g.integers(0, 4, (2, 16, d), dtype=np.uint8),
        "sigma": g.integers(0, 2, (2, 16, d), dtype=np.uint8),
        "vq": g.integers(0, 16, (2, 16, d), dtype=np.uint8),
        "vs": g.standard_normal((2, 16, d // 32)).astype(np.float16),
        "vmn": g.standard_normal((2, 16, d // 32)).astype(np.float16),
        "n_k": g.standard_normal((2, 16)).astype(np.float16),
        "n_r": g.standard_normal((2, 16)).astype(np.float16),
    }
    t = layout.pack_main_tiles(f["idx"], f["sigma"], f["vq"], f["vs"], f["vmn"], f["n_k"], f["n_r"], 4)
    assert t.shape == (2, layout.main_tile_bytes(d, 4)) and layout.main_tile_bytes(d, 4) == 16 * d + 64
    assert layout.main_value_bits(t.shape[-1], d) == 4
    back = layout.unpack_main_tiles(t, d)
    for k, v in f.items():
        assert np.array_equal(back[k].view(np.uint8), v.view(np.uint8)), k
    # norms follow the 8d bytes of value codes and the 2d bytes of scale / minimum
    assert np.array_equal(t[1, 16 * d:16 * d + 32].view("<f2"), f["n_k"][1])


@pytest.mark.parametrize("d", [64, 128, 256])
def test_main_tile_round_trip(d):
    g = np.random.default_rng(d)
    f = {
        "idx": g.integers(0, 4, (3, 16, d), dtype=np.uint8),
        "sigma": g.integers(0, 2, (3, 16, d), dtype=np.uint8),
        "vq": g.integers(0, 4, (3, 16, d), dtype=np.uint8),
        "vs": g.standard_normal((3, 16, d // 32)).astype(np.float16),
        "vmn": g.standard_normal((3, 16, d // 32)).astype(np.float16),
        "n_k": g.standard_normal((3, 16)).astype(np.float16),
        "n_r": g.standard_normal((3, 16)).astype(np.float16),
    }
    t = layout.pack_main_tiles(f["idx"], f["sigma"], f["vq"], f["vs"], f["vmn"], f["n_k"], f["n_r"])
    assert t.shape == (3, layout.main_tile_bytes(d))
    back = layout.unpack_main_tiles(t, d)
    for k, v in f.items():
        assert np.array_equal(back[k].view(np.uint8), v.view(np.uint8)), k
    # field placement: norms at the documented offsets
    assert np.array_equal(t[1, 12 * d:12 * d + 32].view("<f2"), f["n_k"][1])
    assert np.array_equal(t[2, 12 * d + 32:].view("<f2"), f["n_r"][2])
    # KH word 0 of token 0 built from idx >> 1 in even/odd split order
    w0 = int(t[0, 0:4].view("<u4")[0])
    want = 0
    for j in range(16):
        for e in range(2):
            want |= int(f["idx"][0, 0, 2 * j + e] >> 1) << (16 * e + j)
    assert w0 == want


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("vbits,kbits", [(2, 8), (3, 8), (4, 8), (3, 4), (4, 4), (3, 5), (4, 5), (3, 2), (2, 2),
                                         (5, 8), (6, 8), (7, 4), (8, 8), (8, 2)])
def test_alt_tile_round_trip(d, vbits, kbits):
    g = np.random.default_rng(d + vbits + kbits)
    f = {
        "kq": g.integers(0, 1 << kbits, (2, 16, d), dtype=np.uint8),
        "ks": g.standard_normal((2, 16, d // 32)).astype(np.float16),
        "kmn": g.standard_normal((2, 16, d // 32)).astype(np.float16),
        "vidx": g.integers(0, 1 << vbits, (2, 16, d), dtype=np.uint8),
        "n_v": g.standard_normal((2, 16)).astype(np.float16),
    }
    t = layout.pack_alt_tiles(f["kq"], f["ks"], f["kmn"], f["vidx"], f["n_v"], vbits, kbits)
    assert t.shape == (2, layout.alt_tile_bytes(d, vbits, kbits))
    back = layout.unpack_alt_tiles(t, d, vbits)
    for k, v in f.items():
        assert np.array_equal(back[k].view(np.uint8), v.view(np.uint8)), k
    if kbits == 8:
        assert np.array_equal(layout.unpack_alt_tiles(t, d)["vidx"], f["vidx"])  # sizes alone suffice
    # key codes: token 3's kbits-bit stream, then the scale/minimum pairs, then the value streams
    krow = kbits * d // 8
    assert np.array_equal(t[0, 3 * krow:4 * krow], _pack_bigint(f["kq"][0, 3], kbits))
    o_vi = 16 * krow + 2 * d
    row_bytes = vbits * d // 8
    row = t[1, o_vi + 5 * row_bytes:o_vi + 6 * row_bytes]
    assert np.array_equal(row, _pack_bigint(f["vidx"][1, 5], vbits))
    # the value norms follow the index stream
    o_n = o_vi + 16 * row_bytes
    assert np.array_equal(t[0, o_n:o_n + 32].view("<f2"), f["n_v"][0])


@pytest.mark.parametrize("d", [64, 512])
@pytest.mark.parametrize("vbits", [2, 3, 4])
def test_alt_tile_round_trip_fp16_keys(d, vbits):
    # keys kept as fp16 (only the values quantised): 2d key bytes per token, no scale/minimum plane
    g = np.random.default_rng(d + vbits)
    k16 = g.standard_normal((2, 16, d)).astype(np.float16)
    vidx = g.integers(0, 1 << vbits, (2, 16, d), dtype=np.uint8)
    nv = g.standard_normal((2, 16)).astype(np.float16)
    t = layout.pack_alt_tiles(k16, None, None, vidx, nv, vbits, 16)
    assert t.shape == (2, 32 * d + 2 * vbits * d + 32) == (2, layout.alt_tile_bytes(d, vbits, 16))
    assert layout.alt_key_bits(t.shape[-1], d, vbits) == 16
    assert np.array_equal(t[1, 3 * 2 * d:4 * 2 * d].view("<f2"), k16[1, 3])  # token 3's keys, little-endian
    back = layout.unpack_alt_tiles(t, d, vbits)
    assert set(back) == {"k16", "vidx", "n_v"}
    assert np.array_equal(back["k16"].view(np.uint16), k16.view(np.uint16))
    assert np.array_equal(back["vidx"], vidx) and np.array_equal(back["n_v"].view(np.uint16), nv.view(np.uint16))
    # the value stream starts right after the keys
    assert np.array_equal(t[0, 32 * d:32 * d + vbits * d // 8], _pack_bigint(vidx[0, 0], vbits))


def test_bytes_per_token_closed_form():
    assert layout.main_bytes_per_token_head(128) == 100
    # 4-bit values: 48 bytes of key bits, 64 of value codes, 16 of group scale/minimum, 4 of norms
    assert layout.main_bytes_per_token_head(128, 4) == 48 + 64 + 16 + 4 == 132
    # 32 + 16 bytes of key bits, 32 bytes of value codes, 4 groups x 4 bytes, 2 norms
    assert 128 * 3 // 8 + 128 * 2 // 8 + 4 * 4 + 2 + 2 == 100
    for d in (64, 128, 256, 512):
        assert layout.alt_bytes_per_token_head(d) == 1.5 * d + 2
        assert layout.main_tile_bytes(d) % 16 == 0 and layout.alt_tile_bytes(d) % 16 == 0
        for vb in (2, 3, 4):
            for kb in (2, 4, 5, 8):
                # kb bits per key code, 4 B per key block of 32, vb bits per value index, one fp16 norm
                assert layout.alt_bytes_per_token_head(d, vb, kb) == kb * d / 8 + 4 * (d // 32) + vb * d / 8 + 2
                assert layout.alt_tile_bytes(d, vb, kb) % 16 == 0
                assert layout.alt_key_bits(layout.alt_tile_bytes(d, vb, kb), d, vb) == kb
            assert layout.alt_value_bits(layout.alt_tile_bytes(d, vb), d) == vb
            # fp16 keys: 2d bytes per token, then the value indices and the norm
            assert layout.alt_bytes_per_token_head(d, vb, 16) == 2 * d + vb * d / 8 + 2
            assert layout.alt_value_bits(layout.alt_tile_bytes(d, vb, 16), d, 16) == vb


def test_memory_table_of_the_benchmark_page():
    """100 B per token-head plus a 128-token fp16 ring reproduces the printed table."""
    for row in golden("kv_memory_table.json")["rows"]:
        n = row["tokens"]
        n_c, n_buf = cache.ring_split(n)
        assert (n_c, n_buf) == (n - 128, 128)
        fp16 = n * 512
        tq = n_c * layout.main_bytes_per_token_head(128) + n_buf * 512
        assert round(fp16 / tq, 1) == row["ratio_printed"]
        assert round(row["fp16_mb"] * tq / fp16) == row["tq_mb"]


def test_vllm_metal_compression_table_reading():
    """K = b*d/8 + 16 B, V = v*d/8 + 8 B per vector reproduces every printed ratio."""
    d = 128
    for row in golden("vllm_metal_compression.json")["rows"]:
        per = row["k_bits"] * d / 8 + 16 + row["v_bits"] * d / 8 + 8
        assert round(2 * d * 2 / per, 2) == row["ratio_printed"]
    # this project's alternate layout (int8 K + 3-bit V) is tighter by 6 B: one fp16 norm per value
    # vector in place of the table's 8 B; the same holds at 2- and 4-bit values
    assert layout.alt_bytes_per_token_head(128) == 194
    for vb in (2, 3, 4):
        assert layout.alt_bytes_per_token_head(128, vb) == (8 * 128 / 8 + 16) + (vb * 128 / 8 + 8) - 6
    # ... and for the table's other key formats (q5_0, q4_0 and uint2 keys with q3_0 values)
    rows = {r["k_quant"]: r for r in golden("vllm_metal_compression.json")["rows"]}
    for name in ("q5_0", "q4_0", "uint2", "int2"):  # int2 (signed codes) has the bytes of uint2
        row = rows[name]
        per = row["k_bits"] * 128 / 8 + 16 + row["v_bits"] * 128 / 8 + 8
        assert layout.alt_bytes_per_token_head(128, row["v_bits"], row["k_bits"]) == per - 6


def test_ring_split():
    assert cache.ring_split(0) == (0, 0)
    assert cache.ring_split(1) == (0, 1)
    assert cache.ring_split(128) == (0, 128)
    assert cache.ring_split(129) == (128, 1)
    assert cache.ring_split(1024) == (896, 128)
    assert cache.ring_split(32768) == (32640, 128)


@pytest.mark.parametrize("vbits", [2, 4])
def test_main_tile_round_trip_2bit_keys(vbits):
    # 2-bit keys: one Lloyd-Max plane (the 1-bit index) and the QJL plane
    d = 128
    g = np.random.default_rng(vbits)
    f = {
        "idx": g.integers(0, 2, (2, 16, d), dtype=np.uint8),
        "sigma": g.integers(0, 2, (2, 16, d), dtype=np.uint8),
        "vq": g.integers(0, 1 << vbits, (2, 16, d), dtype=np.uint8),
        "vs": g.standard_normal((2, 16, d // 32)).astype(np.float16),
        "vmn": g.standard_normal((2, 16, d // 32)).astype(np.float16),
        "n_k": g.standard_normal((2, 16)).astype(np.float16),
        "n_r": g.standard_normal((2, 16)).astype(np.float16),
    }
    t = layout.pack_main_tiles(f["idx"], f["sigma"], f["vq"], f["vs"], f["vmn"], f["n_k"], f["n_r"], vbits, 2)
    assert t.shape[-1] == (6 + 2 * vbits) * d + 64 and layout.main_bits(t.shape[-1], d) == (2, vbits)
    back = layout.unpack_main_tiles(t, d)
    for k, v in f.items():
        assert np.array_equal(back[k].view(np.uint8), v.view(np.uint8)), k
    # the QJL plane follows the single index plane
    assert np.array_equal(t[:, 2 * d:4 * d], layout.pack_main_tiles(
        f["sigma"], f["sigma"], f["vq"], f["vs"], f["vmn"], f["n_k"], f["n_r"], vbits, 2)[:, 0:2 * d])


def test_bytes_per_token_2bit_keys():
    # 16 bytes of index bits + 16 of QJL bits, 32 of value codes, 16 of group scale/minimum, 4 of norms
    assert layout.main_bytes_per_token_head(128, 2, 2) == 16 + 16 + 32 + 16 + 4 == 84
    assert {layout.main_bits(layout.main_tile_bytes(64, vb, kb), 64) for kb in (2, 3) for vb in (2, 4)} == \
        {(2, 2), (2, 4), (3, 2), (3, 4)}


def test_main_tile_round_trip_4bit_keys():
    # 4-bit keys: three Lloyd-Max index planes (high bit first) and the QJL plane
    d = 64
    g = np.random.default_rng(44)
    f = {
        "idx": g.integers(0, 8, (2, 16, d), dtype=np.uint8),
        "sigma": g.integers(0, 2, (2, 16, d), dtype=np.uint8),
        "vq": g.integers(0, 4, (2, 16, d), dtype=np.uint8),
        "vs": g.standard_normal((2, 16, d // 32)).astype(np.float16),
        "vmn": g.standard_normal((2, 16, d // 32)).astype(np.float16),
        "n_k": g.standard_normal((2, 16)).astype(np.float16),
        "n_r": g.standard_normal((2, 16)).astype(np.float16),
    }
    t = layout.pack_main_tiles(f["idx"], f["sigma"], f["vq"], f["vs"], f["vmn"], f["n_k"], f["n_r"], 2, 4)
    assert t.shape[-1] == 14 * d + 64 and layout.main_bits(t.shape[-1], d, 4) == (4, 2)
    back = layout.unpack_main_tiles(t, d, 4)
    for k, v in f.items():
        assert np.array_equal(back[k].view(np.uint8), v.view(np.uint8)), k
    # plane 0 holds the high index bit
    hi = layout.pack_main_tiles(f["idx"] >> 2, f["sigma"], f["vq"], f["vs"], f["vmn"], f["n_k"], f["n_r"], 2, 2)
    assert np.array_equal(t[:, :2 * d], hi[:, :2 * d])
    assert layout.main_bytes_per_token_head(128, 2, 4) == 64 + 32 + 16 + 4 == 116
