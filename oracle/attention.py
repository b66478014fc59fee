"""Decode attention over the compressed cache plus the exact recent buffer (oracle).

One decode step: every query head h of sequence b attends to all tokens of
its KV head h // n_rep (GQA, "TurboQuant-MLX overview", GPU kernel section:
n_rep instead of repeating K/V), i.e. to the n_c compressed tokens and the
n_buf exact fp16 tokens of the recent buffer ("turboquant-bench": the newest
128 tokens stay fp16; turboquant vLLM guide, §三 hybrid mode: compressed
history plus exact recent buffer), with logits q.k / sqrt(d) and a plain
softmax.  float64 throughout; the caller rounds to float32.

Main layout, compressed logits (the estimator form the fused kernels use,
"TurboQuant-MLX overview", pre-rotated q scoring; turboquant vLLM guide, §二
step 3, unbiased inner-product estimate):

    q_r = H (D q) / sqrt(d),   t = S q_r
    <q, k_hat> = n_k * ( <q_r, c[idx]> + sqrt(pi/2)/m * n_r * <t, 2 sigma - 1> )

``decode_main_bruteforce`` instead rebuilds every k_hat explicitly and is
used only to pin the estimator form.

Alternate layout: k_hat = mn + s * code per 32-block (no rotation) and
v_hat = n_v * D H c[idx] / sqrt(d).
"""
from __future__ import annotations

import numpy as np

from . import cache, quant, rotation


def _softmax_combine(logits: np.ndarray, values: np.ndarray) -> np.ndarray:
    """logits [H, T], values [T, d] -> [H, d] (T may be 0 -> zeros)."""
    if logits.shape[-1] == 0:
        return np.zeros((logits.shape[0], values.shape[-1]))
    m = logits.max(axis=-1, keepdims=True)
    p = np.exp(logits - m)
    return (p @ values) / p.sum(axis=-1, keepdims=True)


def _ring(ring_k, ring_v, b, kvh, n):
    if n == 0:
        return None, None
    return (np.asarray(ring_k[b, kvh, :n], dtype=np.float64),
            np.asarray(ring_v[b, kvh, :n], dtype=np.float64))


def decode_main(q16, pool, block_table, n_c, ring_k, ring_v, n_buf, signs, centroids, s_mat, n_kv):
    """Main-layout decode step; returns float64 [B, Hq, d]."""
    q16 = np.asarray(q16, dtype=np.float16)
    bsz, hq, d = q16.shape
    n_rep = hq // n_kv
    m = s_mat.shape[0]
    c = np.asarray(centroids, dtype=np.float64)
    s64 = np.asarray(s_mat, dtype=np.float64)
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        nc = int(n_c[b])
        nb = int(n_buf[b])
        f = cache.read_main(pool, block_table, b, nc, d, cache.key_bits_of(centroids)) if nc else None
        for g in range(n_kv):
            q = q16[b, g * n_rep:(g + 1) * n_rep].astype(np.float64)
            logits = []
            vals = []
            if nc:
                q_r = rotation.rotate(q, signs)
                t = q_r @ s64.T
                pm = 2.0 * f["sigma"][g].astype(np.float64) - 1.0
                lm = q_r @ c[f["idx"][g]].T
                qjl = t @ pm.T
                nk = f["n_k"][g].astype(np.float64)
                nr = f["n_r"][g].astype(np.float64)
                logits.append(nk * (lm + (quant.QJL_SCALE / m) * nr * qjl) / np.sqrt(d))
                vals.append(quant.group_dequant(f["vq"][g], f["vs"][g], f["vmn"][g], 32))
            kr, vr = _ring(ring_k, ring_v, b, g, nb)
            if kr is not None:
                logits.append(q @ kr.T / np.sqrt(d))
                vals.append(vr)
            lg = np.concatenate(logits, axis=-1) if logits else np.zeros((n_rep, 0))
            vv = np.concatenate(vals, axis=0) if vals else np.zeros((0, d))
            out[b, g * n_rep:(g + 1) * n_rep] = _softmax_combine(lg, vv)
    return out


def decode_main_bruteforce(q16, pool, block_table, n_c, ring_k, ring_v, n_buf, signs, centroids, s_mat, n_kv):
    """softmax(q K_hat^T / sqrt(d)) V_hat with every k_hat rebuilt explicitly (small inputs only)."""
    q16 = np.asarray(q16, dtype=np.float16)
    bsz, hq, d = q16.shape
    n_rep = hq // n_kv
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        nc = int(n_c[b])
        nb = int(n_buf[b])
        f = cache.read_main(pool, block_table, b, nc, d, cache.key_bits_of(centroids)) if nc else None
        for h in range(hq):
            g = h // n_rep
            q = q16[b, h].astype(np.float64)
            keys = []
            vals = []
            for tok in range(nc):
                enc = {key: f[key][g, tok] for key in ("n_k", "idx", "n_r", "sigma")}
                keys.append(quant.dequant_keys(enc, signs, centroids, s_mat))
                vals.append(quant.group_dequant(f["vq"][g, tok], f["vs"][g, tok], f["vmn"][g, tok], 32))
            for tok in range(nb):
                keys.append(np.asarray(ring_k[b, g, tok], dtype=np.float64))
                vals.append(np.asarray(ring_v[b, g, tok], dtype=np.float64))
            if not keys:
                continue
            kk = np.stack(keys)
            vv = np.stack(vals)
            logit = kk @ q / np.sqrt(d)
            p = np.exp(logit - logit.max())
            out[b, h] = p @ vv / p.sum()
    return out


def decode_alt(q16, pool, block_table, n_c, ring_k, ring_v, n_buf, signs, centroids3, n_kv):
    """Alternate-layout decode step; returns float64 [B, Hq, d]."""
    q16 = np.asarray(q16, dtype=np.float16)
    bsz, hq, d = q16.shape
    n_rep = hq // n_kv
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        nc = int(n_c[b])
        nb = int(n_buf[b]) if n_buf is not None else 0
        f = cache.read_alt(pool, block_table, b, nc, d, cache.value_bits_of(centroids3)) if nc else None
        for g in range(n_kv):
            q = q16[b, g * n_rep:(g + 1) * n_rep].astype(np.float64)
            logits = []
            vals = []
            if nc:
                khat = quant.alt_keys({key: val[g] for key, val in f.items()})
                logits.append(q @ khat.T / np.sqrt(d))
                vals.append(quant.dequant_alt_values(f["vidx"][g], f["n_v"][g], signs, centroids3))
            kr, vr = _ring(ring_k, ring_v, b, g, nb) if nb else (None, None)
            if kr is not None:
                logits.append(q @ kr.T / np.sqrt(d))
                vals.append(vr)
            lg = np.concatenate(logits, axis=-1) if logits else np.zeros((n_rep, 0))
            vv = np.concatenate(vals, axis=0) if vals else np.zeros((0, d))
            out[b, g * n_rep:(g + 1) * n_rep] = _softmax_combine(lg, vv)
    return out


def attend_exact(q16, k16, v16, n_kv):
    """Plain fp16-input attention of q [B, Hq, d] over k, v [B, Hkv, T, d] (float64)."""
    q = np.asarray(q16, dtype=np.float64)
    k = np.asarray(k16, dtype=np.float64)
    v = np.asarray(v16, dtype=np.float64)
    bsz, hq, d = q.shape
    n_rep = hq // n_kv
    out = np.zeros((bsz, hq, d))
    for b in range(bsz):
        for h in range(hq):
            g = h // n_rep
            out[b, h] = _softmax_combine((k[b, g] @ q[b, h] / np.sqrt(d))[None, :], v[b, g])[0]
    return out
