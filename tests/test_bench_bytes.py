"""The bench's algorithmic bytes per token-head against the oracle's page layouts (no GPU).

The roofline numerator of every workload counts records of the size the oracle's tiles fix
(tile bytes / 16 tokens), at the workload's key and value widths.
"""
import bench
from oracle import layout


def test_record_bytes_equal_oracle_tiles():
    for name, w in bench.WORKLOADS.items():
        d = w["d"]
        if w["layout"] == "main":
            tile = layout.main_tile_bytes(d, w.get("vbits", 2), w.get("kbits", 3))
        else:
            tile = layout.alt_tile_bytes(d, w.get("vbits", 3), w.get("kbits", 8))
        assert bench.record_bytes(w) * layout.P == tile, name


def test_step_bytes_closed_form():
    # the default widths: 100 B per compressed token-head, 4d B per ring token-head, q + out
    w = dict(bench.WORKLOADS["qwen3-0.6b-32k"])
    assert bench.record_bytes(w) == 100
    got = bench.step_bytes(w, [32769])
    assert got == 4 * (32768 * 100 + 1 * 512) + 16 * 128 * 6
    a = dict(bench.WORKLOADS["alt-d128"])
    assert bench.step_bytes(a, [65536] * 4) == 4 * 8 * 65536 * 194 + 4 * 8 * 128 * 6


def test_ncu_traffic_is_used_only_for_the_captured_sources(tmp_path, monkeypatch):
    """roofline.traffic: the DRAM bytes of a listed ncu capture, returned only while every source
    file the capture names still has the recorded sha256; any mismatch, a missing file, another
    kernel or workload gives None."""
    import hashlib
    import json
    import os

    csrc = tmp_path / "kv_cache_quantization_tq_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cu").write_bytes(b"kernel source")
    (csrc / "b.cuh").write_bytes(b"header")
    digest = {f: hashlib.sha256((csrc / f).read_bytes()).hexdigest() for f in ("a.cu", "b.cuh")}
    table = {"w1": {"kernel": "k1", "dram_bytes": 1234, "capture": "...", "sources": digest}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(table))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("w1", "k1") == 1234
    assert bench.ncu_traffic("w1", "k2") is None  # another kernel
    assert bench.ncu_traffic("w2", "k1") is None  # another workload
    (csrc / "b.cuh").write_bytes(b"header, edited")
    assert bench.ncu_traffic("w1", "k1") is None  # a source changed since the capture
    os.remove(csrc / "b.cuh")
    assert bench.ncu_traffic("w1", "k1") is None  # a source is gone
