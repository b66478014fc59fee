"""Encoders of the compressed KV cache (oracle).

Main layout (3-bit keys, 2-bit values):

* key, per (token, KV head) vector k of dimension d (turboquant vLLM guide,
  §二 steps 1-3; "turboquant-bench" compression details: rotation +
  Lloyd-Max codebook + QJL sign sketch):
    n_k   = ||k||, stored as fp16
    u     = k / ||k||   (u = 0 when ||k|| = 0)
    y     = H (D u) / sqrt(d)
    idx_i = number of codebook boundaries b_j with b_j <= y_i (ties go up)
    r     = y - c[idx]
    n_r   = ||r||, stored as fp16
    z     = S r             (S: m x d Gaussian, m = d)
    sigma_j = 1 if z_j >= 0 else 0
* value, per group of 32 consecutive coordinates ("turboquant-bench"
  compression details: asymmetric group quantisation, per-group min and max,
  2 bits per value), in IEEE float32:
    mn = min, mx = max over the group (fp16 inputs are exact in fp32)
    s  = fp16((mx - mn) / 3)
    q  = clamp(rint((v - mn) / s), 0, 3) with round-half-even, q = 0 if s == 0

Alternate layout (vllm-metal TurboQuant guide, quantisation principle table:
K per-block affine without rotation, V Walsh-Hadamard rotation + Lloyd-Max):

* key: the same asymmetric quantiser with 255 levels on blocks of 32 (8-bit
  codes, fp16 scale and minimum);
* value: n_v = fp16(||v||), y = H (D v/||v||) / sqrt(d), 3-bit Lloyd-Max
  index of every coordinate (8 centroids).

Dequantised forms used by the decode oracle:
    k_hat = n_k * D H (c[idx] + sqrt(pi/2)/m * n_r * S^T (2 sigma - 1)) / sqrt(d)
    v_hat = mn + s * q
    v_hat(alt) = n_v * D H c[idx] / sqrt(d)
"""
from __future__ import annotations

import numpy as np

from . import rotation

QJL_SCALE = np.sqrt(np.pi / 2.0)


def assign(y: np.ndarray, boundaries: np.ndarray) -> np.ndarray:
    """Lloyd-Max index = count of boundaries <= y (ties go to the upper cell)."""
    return np.searchsorted(np.asarray(boundaries, dtype=np.float64), y, side="right").astype(np.uint8)


def boundaries_of(centroids: np.ndarray) -> np.ndarray:
    c = np.asarray(centroids, dtype=np.float64)
    return 0.5 * (c[:-1] + c[1:])


def encode_keys(k16: np.ndarray, signs: np.ndarray, centroids: np.ndarray, s_mat: np.ndarray):
    """Encode fp16 keys [..., d].

    Returns a dict with the stored fields ``n_k`` (fp16), ``idx`` (uint8),
    ``n_r`` (fp16), ``sigma`` (uint8 0/1) and, for boundary checks, the
    float64 intermediates ``y`` (rotated unit key) and ``z`` (= S r).
    """
    k = np.asarray(k16, dtype=np.float16).astype(np.float64)
    c = np.asarray(centroids, dtype=np.float64)
    nk = np.sqrt(np.sum(k * k, axis=-1))
    safe = np.where(nk > 0, nk, 1.0)
    u = np.where(nk[..., None] > 0, k / safe[..., None], 0.0)
    y = rotation.rotate(u, signs)
    idx = assign(y, boundaries_of(c))
    r = y - c[idx]
    nr = np.sqrt(np.sum(r * r, axis=-1))
    z = r @ np.asarray(s_mat, dtype=np.float64).T
    sigma = (z >= 0).astype(np.uint8)
    return {
        "n_k": nk.astype(np.float16),
        "idx": idx,
        "n_r": nr.astype(np.float16),
        "sigma": sigma,
        "y": y,
        "z": z,
        "n_k_exact": nk,
        "n_r_exact": nr,
    }


def inner_product_estimate(q, n_k, idx, n_r, sigma, signs, centroids, s_mat):
    """Estimator of <q, k> from one encoded key (float64).

    n_k * (<q_r, c[idx]> + sqrt(pi/2)/m * n_r * <S q_r, 2 sigma - 1>), q_r = H (D q)/sqrt(d).
    """
    q = np.asarray(q, dtype=np.float64)
    c = np.asarray(centroids, dtype=np.float64)
    s64 = np.asarray(s_mat, dtype=np.float64)
    m = s64.shape[0]
    q_r = rotation.rotate(q, signs)
    t = q_r @ s64.T
    pm = 2.0 * np.asarray(sigma, dtype=np.float64) - 1.0
    lm = np.sum(q_r * c[idx], axis=-1)
    qjl = np.sum(t * pm, axis=-1)
    return np.asarray(n_k, np.float64) * (lm + (QJL_SCALE / m) * np.asarray(n_r, np.float64) * qjl)


def group_quant(x16: np.ndarray, group: int, levels: int):
    """Asymmetric min/max quantiser in IEEE float32.

    x16: fp16 [..., n] with n a multiple of ``group``.
    Returns (codes uint8 [..., n], scale fp16 [..., n/group], minimum fp16 [..., n/group]).
    """
    x = np.asarray(x16, dtype=np.float16).astype(np.float32)
    shape = x.shape
    g = x.reshape(shape[:-1] + (shape[-1] // group, group))
    mn = g.min(axis=-1, keepdims=True)
    mx = g.max(axis=-1, keepdims=True)
    s16 = ((mx - mn) / np.float32(levels)).astype(np.float16)
    s = s16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.rint((g - mn) / s)
    q = np.where(s > 0, np.clip(qf, 0, levels), 0).astype(np.uint8)
    return q.reshape(shape), s16[..., 0], mn.astype(np.float16)[..., 0]


def signed_group_quant(x16: np.ndarray, group: int, levels: int):
    """Signed symmetric mid-rise quantiser in IEEE float32 (this library's reading of the vllm-metal
    guide's int2 key format, beside the affine uint2): per group, a = max |x|,
    s = fp16(a / (levels / 2)), mn = fp16(-(levels / 2) s), q = clamp(rint((x - mn) / s), 0, levels)
    with round-half-even, q = 0 if s == 0.  The levels mn + s q are (q - levels / 2) s up to the fp16
    rounding of mn.  Returns (codes, scale fp16, minimum fp16) like group_quant."""
    x = np.asarray(x16, dtype=np.float16).astype(np.float32)
    shape = x.shape
    g = x.reshape(shape[:-1] + (shape[-1] // group, group))
    half = np.float32(levels) / np.float32(2)
    a = np.abs(g).max(axis=-1, keepdims=True)
    s16 = (a / half).astype(np.float16)
    s = s16.astype(np.float32)
    mn16 = (-half * s).astype(np.float16)
    mn = mn16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.rint((g - mn) / s)
    q = np.where(s > 0, np.clip(qf, 0, levels), 0).astype(np.uint8)
    return q.reshape(shape), s16[..., 0], mn16[..., 0]


def group_dequant(q: np.ndarray, scale16: np.ndarray, min16: np.ndarray, group: int) -> np.ndarray:
    """mn + s * q in float64."""
    q = np.asarray(q, dtype=np.float64)
    shape = q.shape
    g = q.reshape(shape[:-1] + (shape[-1] // group, group))
    out = min16.astype(np.float64)[..., None] + scale16.astype(np.float64)[..., None] * g
    return out.reshape(shape)


def encode_values(v16: np.ndarray, group: int = 32, bits: int = 2):
    """Main-layout values: ``bits``-bit codes (2 or 4; turboquant vLLM guide, --value-bits),
    fp16 scale, fp16 minimum per group."""
    return group_quant(v16, group, (1 << bits) - 1)


def dequant_keys(enc: dict, signs: np.ndarray, centroids: np.ndarray, s_mat: np.ndarray) -> np.ndarray:
    """Explicit reconstruction k_hat of main-layout keys (float64)."""
    c = np.asarray(centroids, dtype=np.float64)
    m = s_mat.shape[0]
    pm = 2.0 * enc["sigma"].astype(np.float64) - 1.0
    corr = pm @ np.asarray(s_mat, dtype=np.float64)
    x = c[enc["idx"]] + (QJL_SCALE / m) * enc["n_r"].astype(np.float64)[..., None] * corr
    return enc["n_k"].astype(np.float64)[..., None] * rotation.unrotate(x, signs)


def encode_alt_keys(k16: np.ndarray, block: int = 32, bits: int = 8, signed: bool = False):
    """Alternate-layout keys: bits-bit affine codes per block of 32 (2^bits - 1 steps), or with
    signed=True (2 bits only: int2) the signed symmetric mid-rise codes of signed_group_quant.  With
    16 bits the keys stay as they are (fp16): only the values are quantised (the V-only mode of the
    "TurboQuant-MLX overview", usage paths)."""
    if bits == 16:
        return np.asarray(k16, dtype=np.float16), None, None
    if signed:
        assert bits == 2, "signed keys are the 2-bit int2 format"
        return signed_group_quant(k16, block, 3)
    return group_quant(k16, block, (1 << bits) - 1)


def alt_keys(fields) -> np.ndarray:
    """Keys of unpacked alternate-layout tiles in float64: the fp16 keys, or mn + s q."""
    if "k16" in fields:
        return np.asarray(fields["k16"], dtype=np.float64)
    return group_dequant(fields["kq"], fields["ks"], fields["kmn"], 32)


def encode_alt_values(v16: np.ndarray, signs: np.ndarray, centroids: np.ndarray):
    """Alternate-layout values: (idx uint8 Lloyd-Max index, n_v fp16, y float64)."""
    v = np.asarray(v16, dtype=np.float16).astype(np.float64)
    nv = np.sqrt(np.sum(v * v, axis=-1))
    safe = np.where(nv > 0, nv, 1.0)
    u = np.where(nv[..., None] > 0, v / safe[..., None], 0.0)
    y = rotation.rotate(u, signs)
    idx = assign(y, boundaries_of(centroids))
    return {"idx": idx, "n_v": nv.astype(np.float16), "y": y}


def dequant_alt_values(idx: np.ndarray, nv16: np.ndarray, signs: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    c = np.asarray(centroids, dtype=np.float64)
    return nv16.astype(np.float64)[..., None] * rotation.unrotate(c[idx], signs)
