"""Pins for the oracle's key/value encoders."""
import math

import numpy as np
import pytest

import synth
from oracle import codebook, quant, rng, rotation


def _brute_group_codes(x16, group, levels):
    """Nearest level index by explicit search over all levels (ties to even), float32."""
    x = np.asarray(x16, np.float16).astype(np.float32).ravel()
    out = np.zeros(x.size, np.uint8)
    for g0 in range(0, x.size, group):
        blk = x[g0:g0 + group]
        mn = np.float32(blk.min())
        mx = np.float32(blk.max())
        s = np.float32(np.float16(np.float32(mx - mn) / np.float32(levels)))
        for i, v in enumerate(blk):
            if s == 0:
                continue
            t = np.float32(np.float32(v - mn) / s)
            best, bd = 0, None
            for q in range(levels + 1):
                dist = abs(float(t) - q)
                if bd is None or dist < bd - 1e-12 or (abs(dist - bd) <= 1e-12 and q % 2 == 0):
                    best, bd = q, dist
            out[g0 + i] = best
    return out


@pytest.mark.parametrize("levels", [3, 15, 31, 255])
def test_group_quant_brute_force(levels):
    g = np.random.default_rng(levels)
    x = (g.standard_normal((6, 64)) * g.lognormal(size=(6, 1))).astype(np.float16)
    x[0, :32] = np.float16(1.5)  # constant group -> scale 0 -> all codes 0
    x[1, :4] = [0, 1, 2, 3]      # exact levels
    q, s, mn = quant.group_quant(x, 32, levels)
    assert np.array_equal(q.ravel(), _brute_group_codes(x, 32, levels))
    assert s[0, 0] == 0 and np.all(q[0, :32] == 0)
    # reconstruction error bounded by half a step (plus rounding slack)
    rec = quant.group_dequant(q, s, mn, 32)
    step = np.repeat(s.astype(np.float64), 32, axis=-1)
    assert np.all(np.abs(rec - x.astype(np.float64)) <= 0.5 * step + 1e-3 * step + 1e-7)


def test_group_quant_hand_worked():
    v = np.zeros(32, np.float16)
    v[:6] = [0.0, 1.0, 2.0, 3.0, 1.5, 0.5]
    q, s, mn = quant.group_quant(v, 32, 3)
    assert float(s[0]) == 1.0 and float(mn[0]) == 0.0
    # 1.5 and 0.5 are exact ties: round half to even -> 2 and 0
    assert q[:6].tolist() == [0, 1, 2, 3, 2, 0]


def _tables(seed, d, bits=2):
    c, _ = codebook.lloyd_max(d, bits)
    return rng.signs(seed, d), c, rng.gaussian_matrix(seed, d, d)


def test_key_encoder_fields():
    d = 128
    sg, c, s = _tables(0, d)
    k, _ = synth.kv_main(0, 1, 1, 64, d)
    k = k[0, 0]
    k[3] = 0  # zero key
    enc = quant.encode_keys(k, sg, c, s)
    kf = k.astype(np.float64)
    assert np.array_equal(enc["n_k"], np.linalg.norm(kf, axis=1).astype(np.float16))
    y = enc["y"]
    nz = np.linalg.norm(kf, axis=1) > 0
    assert np.allclose(np.linalg.norm(y[nz], axis=1), 1.0, atol=1e-12)
    # nearest centroid by brute force (no exact ties in random data)
    assert np.array_equal(enc["idx"][nz], np.argmin(np.abs(y[nz][..., None] - c), axis=-1))
    r = y - c[enc["idx"]]
    assert np.array_equal(enc["n_r"], np.linalg.norm(r, axis=1).astype(np.float16))
    assert np.array_equal(enc["sigma"], (r @ s.astype(np.float64).T >= 0).astype(np.uint8))
    # zero key: y = 0 lies on the middle boundary and goes up
    assert np.all(enc["idx"][3] == 2) and enc["n_k"][3] == 0
    # a sketch row of zeros gives z_j = 0 exactly, which counts as a positive sign
    s0 = s.copy()
    s0[5] = 0
    assert np.all(quant.encode_keys(k, sg, c, s0)["sigma"][:, 5] == 1)


def test_tie_goes_to_upper_cell_and_sign_of_zero():
    b = np.array([-0.1, 0.0, 0.1])
    assert quant.assign(np.array([-0.1, 0.0, 0.1, 0.05]), b).tolist() == [1, 2, 3, 2]


def test_estimator_equals_dequantised_inner_product():
    d = 128
    sg, c, s = _tables(4, d)
    k, _ = synth.kv_main(4, 1, 1, 32, d)
    q = synth.queries(4, 1, 1, d)[0, 0]
    enc = quant.encode_keys(k[0, 0], sg, c, s)
    est = quant.inner_product_estimate(q, enc["n_k"], enc["idx"], enc["n_r"], enc["sigma"], sg, c, s)
    khat = quant.dequant_keys(enc, sg, c, s)
    assert np.allclose(est, khat @ q.astype(np.float64), rtol=1e-12, atol=1e-10)


def test_qjl_estimator_unbiased_over_seeds():
    """Mean over 10k seeds of the estimate of <q, k> is within 3 SE of the truth."""
    d = 128
    g = np.random.default_rng(11)
    k = g.standard_normal(d)
    q = 0.6 * k + g.standard_normal(d)
    true = float(q @ k)
    c, _ = codebook.lloyd_max(d, 2)
    n = 10_000
    est = np.empty(n)
    est_lm = np.empty(n)
    for seed in range(n):
        sg = rng.signs(seed, d)
        s = rng.gaussian_matrix(seed, d, d)
        enc = quant.encode_keys(k.astype(np.float16), sg, c, s)
        est[seed] = quant.inner_product_estimate(q, enc["n_k_exact"], enc["idx"], enc["n_r_exact"], enc["sigma"], sg, c, s)
        est_lm[seed] = enc["n_k_exact"] * np.dot(rotation.rotate(q, sg), c[enc["idx"]])
    true16 = float(q @ k.astype(np.float16).astype(np.float64))
    se = est.std(ddof=1) / math.sqrt(n)
    assert abs(est.mean() - true16) < 3 * se, (est.mean(), true16, se)
    # without the QJL term the Lloyd-Max part alone is biased (shrinks the inner product)
    se_lm = est_lm.std(ddof=1) / math.sqrt(n)
    assert abs(est_lm.mean() - true16) > 10 * max(se_lm, se)
    assert abs(true - true16) < 1e-2


@pytest.mark.parametrize("lm_bits", [1, 3])
def test_qjl_estimator_unbiased_at_other_key_widths(lm_bits):
    """The same unbiasedness with 1- and 3-bit Lloyd-Max indices (2- and 4-bit keys, turboquant vLLM
    guide, --key-bits): the QJL term removes the bias of any codebook, d = 64, 10k seeds."""
    d = 64
    g = np.random.default_rng(12 + lm_bits)
    k = g.standard_normal(d)
    q = 0.5 * k + g.standard_normal(d)
    c, _ = codebook.lloyd_max(d, lm_bits)
    n = 10_000
    est = np.empty(n)
    est_lm = np.empty(n)
    for seed in range(n):
        sg = rng.signs(seed, d)
        s = rng.gaussian_matrix(seed, d, d)
        enc = quant.encode_keys(k.astype(np.float16), sg, c, s)
        est[seed] = quant.inner_product_estimate(q, enc["n_k_exact"], enc["idx"], enc["n_r_exact"], enc["sigma"], sg, c, s)
        est_lm[seed] = enc["n_k_exact"] * np.dot(rotation.rotate(q, sg), c[enc["idx"]])
    true16 = float(q @ k.astype(np.float16).astype(np.float64))
    se = est.std(ddof=1) / math.sqrt(n)
    assert abs(est.mean() - true16) < 3 * se, (est.mean(), true16, se)
    se_lm = est_lm.std(ddof=1) / math.sqrt(n)
    assert abs(est_lm.mean() - true16) > 10 * max(se_lm, se)  # the Lloyd-Max part alone shrinks it


def test_alt_value_encoder():
    d = 256
    sg = rng.signs(2, d)
    c3, _ = codebook.lloyd_max(d, 3)
    _, v = synth.kv_alt(2, 1, 1, 40, d)
    enc = quant.encode_alt_values(v[0, 0], sg, c3)
    y = enc["y"]
    assert np.array_equal(enc["idx"], np.argmin(np.abs(y[..., None] - c3), axis=-1))
    vhat = quant.dequant_alt_values(enc["idx"], enc["n_v"], sg, c3)
    vf = v[0, 0].astype(np.float64)
    cos = np.sum(vhat * vf, axis=1) / np.linalg.norm(vhat, axis=1) / np.linalg.norm(vf, axis=1)
    assert np.all(cos > 0.97)
    # dequantised vector has norm n_v * ||c[idx]||
    assert np.allclose(np.linalg.norm(vhat, axis=1),
                       enc["n_v"].astype(np.float64) * np.linalg.norm(c3[enc["idx"]], axis=1), rtol=1e-12)


def test_signed_group_quant_int2():
    """int2 keys (signed symmetric mid-rise, this library's reading): s = fp16(max|x| / 1.5),
    mn = fp16(-1.5 s), codes = the nearest of the four levels mn + s c (brute force, ties to even)."""
    g = np.random.default_rng(5)
    x = (g.standard_normal((5, 64)) * g.lognormal(size=(5, 1))).astype(np.float16)
    x[0, :32] = 0                        # zero block -> scale 0, codes 0
    x[1, 32:64] = np.abs(x[1, 32:64])    # one-signed block: the symmetric range still spans +-max
    q, s, mn = quant.signed_group_quant(x, 32, 3)
    xf = x.astype(np.float32).reshape(5, 2, 32)
    a = np.abs(xf).max(axis=-1)
    assert np.array_equal(s, (a / np.float32(1.5)).astype(np.float16))
    assert np.array_equal(mn, (np.float32(-1.5) * s.astype(np.float32)).astype(np.float16))
    assert s[0, 0] == 0 and np.all(q[0, :32] == 0)
    # the same codes as the brute-force nearest level of the affine form with these (s, mn)
    qq = q.reshape(5, 2, 32)
    for r in range(5):
        for b in range(2):
            sf, mf = np.float32(s[r, b]), np.float32(mn[r, b])
            for i in range(32):
                if sf == 0:
                    continue
                t = np.float32(np.float32(xf[r, b, i] - mf) / sf)
                d = [abs(float(t) - c) for c in range(4)]
                best = min(range(4), key=lambda c: (round(d[c], 12), c % 2))
                assert qq[r, b, i] == best
    # levels symmetric about zero up to the fp16 rounding of mn; the block maximum takes the top code
    lv_lo = mn.astype(np.float64)
    lv_hi = mn.astype(np.float64) + 3 * s.astype(np.float64)
    assert np.all(np.abs(lv_lo + lv_hi) <= np.abs(lv_hi) * 2.0 ** -10 + 1e-12)
    top = np.argmax(np.abs(xf), axis=-1)
    sign = np.take_along_axis(xf, top[..., None], -1)[..., 0]
    code = np.take_along_axis(qq, top[..., None], -1)[..., 0]
    nz = s.astype(np.float32) > 0
    assert np.all(code[nz & (sign > 0)] == 3) and np.all(code[nz & (sign < 0)] == 0)
    # the one-signed block: no code below the middle (all values >= 0 sit at the upper levels)
    assert np.all(qq[1, 1] >= 1)
