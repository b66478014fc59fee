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
