"""Python binding of libtq (ctypes): argument marshalling only.

Every name mirrors a C entry point of ``include/tq.h``; all arithmetic runs
in the library's CUDA kernels (device calls) or in its host C++ (setup and
host packing).  Device arrays are torch CUDA tensors; their data pointers
and the current torch CUDA stream are handed to the library unchanged.  If
``libtq.so`` is missing the import fails loudly: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE, TQ_ERR_CUDA = range(5)
TQ_LAYOUT_MAIN, TQ_LAYOUT_ALT = 0, 1
TQ_DEVERR_BLOCK_ID, TQ_DEVERR_POSITION, TQ_DEVERR_RING, TQ_DEVERR_CHUNKS, TQ_DEVERR_TIMEOUT = 1, 2, 4, 8, 16
TQ_DECODE_AUTO, TQ_DECODE_MMA_SYNC, TQ_DECODE_TCGEN05 = 0, 1, 2
TQ_KEY_AFFINE, TQ_KEY_SIGNED = 0, 1


class TQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.tq_status_string(status).decode()}")


class tq_config(C.Structure):
    _fields_ = [
        ("head_dim", C.c_int),
        ("num_q_heads", C.c_int),
        ("num_kv_heads", C.c_int),
        ("page_size", C.c_int),
        ("ring_capacity", C.c_int),
        ("layout", C.c_int),
        ("key_bits", C.c_int),
        ("value_bits", C.c_int),
        ("group_size", C.c_int),
        ("qjl_m", C.c_int),
        ("seed", C.c_uint64),
        ("key_format", C.c_int),
    ]


class tq_profile(C.Structure):
    _fields_ = [
        ("decode_launches", C.c_int64),
        ("decode_ms", C.c_double),
        ("encode_launches", C.c_int64),
        ("encode_ms", C.c_double),
        ("merge_launches", C.c_int64),
        ("merge_ms", C.c_double),
        ("decode_kernel", C.c_char_p),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtq.so is not built ({LIB_PATH}); run kv_cache_quantization_tq_gb300.build.build()")
    return C.CDLL(LIB_PATH)


lib = _load()

_vp, _i, _i64, _u64, _sz = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_size_t
_SIGS = {
    "tq_status_string": (C.c_char_p, [_i]),
    "tq_config_init": (_i, [C.POINTER(tq_config), _i, _i, _i, _i, _u64]),
    "tq_config_check": (_i, [C.POINTER(tq_config), C.POINTER(_sz)]),
    "tq_create": (_i, [C.POINTER(tq_config), C.POINTER(_vp)]),
    "tq_create_with_tables": (_i, [C.POINTER(tq_config), _vp, _vp, _vp, C.POINTER(_vp)]),
    "tq_destroy": (None, [_vp]),
    "tq_get_tables": (_i, [_vp, _vp, _vp, _vp, _vp]),
    "tq_lloyd_max": (_i, [_i, _i, _vp, _vp]),
    "tq_generate_tables": (_i, [_u64, _i, _i, _vp, _vp]),
    "tq_bytes_per_token_head": (_sz, [_vp]),
    "tq_page_bytes": (_sz, [_vp]),
    "tq_workspace_size": (_i, [_vp, _i, _i, C.POINTER(_sz)]),
    "tq_encode_flush": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _i, _vp, _i, _vp]),
    "tq_append_token": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _vp, _i, _vp]),
    "tq_decode_attention": (_i, [_vp, _vp, _i, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _i, _vp, _vp, _sz, _vp]),
    "tq_decode_attention_static": (_i, [_vp, _vp, _i, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _i, _vp, _vp]),
    "tq_dequantize": (_i, [_vp, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp]),
    "tq_dequantize_bf16": (_i, [_vp, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp]),
    "tq_should_materialize": (_i, [_i64, _i64, _i, _i, _i64]),
    "tq_pack": (_i, [_vp, _i64, _i, _vp, _vp]),
    "tq_unpack": (_i, [_vp, _i64, _i, _vp, _vp]),
    "tq_pack_host": (_i, [_vp, _i64, _i, _vp]),
    "tq_unpack_host": (_i, [_vp, _i64, _i, _vp]),
    "tq_get_device_errors": (_i, [_vp, C.POINTER(C.c_uint32), _vp]),
    "tq_launch_count": (_i64, [_vp]),
    "tq_set_decode_path": (_i, [_vp, _i]),
    "tq_profile_begin": (_i, [_vp]),
    "tq_profile_end": (_i, [_vp, C.POINTER(tq_profile)]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def _check(st: int, where: str):
    if st != TQ_OK:
        raise TQError(st, where)


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------- host-only calls
def tq_lloyd_max(d: int, bits: int):
    c = np.zeros(1 << bits, np.float64)
    b = np.zeros((1 << bits) - 1, np.float64)
    _check(lib.tq_lloyd_max(d, bits, _np_ptr(c), _np_ptr(b)), "tq_lloyd_max")
    return c, b


def tq_generate_tables(seed: int, d: int, m: int = 0):
    signs = np.zeros(d, np.float32)
    sketch = np.zeros((m, d), np.float32) if m else None
    _check(lib.tq_generate_tables(seed, d, m, _np_ptr(signs), _np_ptr(sketch) if m else None), "tq_generate_tables")
    return signs, sketch


def tq_pack_host(codes: np.ndarray, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    out = np.zeros((codes.size * bits + 7) // 8, np.uint8)
    _check(lib.tq_pack_host(_np_ptr(codes), codes.size, bits, _np_ptr(out)), "tq_pack_host")
    return out


def tq_unpack_host(buf: np.ndarray, n: int, bits: int) -> np.ndarray:
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    out = np.zeros(n, np.uint8)
    _check(lib.tq_unpack_host(_np_ptr(buf), n, bits, _np_ptr(out)), "tq_unpack_host")
    return out


def tq_config_init(layout: int, head_dim: int, num_q_heads: int, num_kv_heads: int, seed: int = 0) -> tq_config:
    cfg = tq_config()
    _check(lib.tq_config_init(C.byref(cfg), layout, head_dim, num_q_heads, num_kv_heads, seed), "tq_config_init")
    return cfg


def tq_should_materialize(history_tokens: int, query_tokens: int, head_dim: int, num_kv_heads: int,
                          max_mib: int = -1) -> bool:
    """The prefill admission rule of the materialisation (host only); ValueError on bad arguments."""
    r = lib.tq_should_materialize(history_tokens, query_tokens, head_dim, num_kv_heads, max_mib)
    if r < 0:
        raise ValueError("tq_should_materialize: negative counts, or head_dim / num_kv_heads <= 0")
    return bool(r)


def tq_config_check(cfg: tq_config) -> int:
    """Bytes per token and KV head of a valid configuration (no CUDA call); TQError otherwise."""
    n = C.c_size_t(0)
    _check(lib.tq_config_check(C.byref(cfg), C.byref(n)), "tq_config_check")
    return n.value


# ---------------------------------------------------------------- device calls
def _stream(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t, dtype=None, name="tensor"):
    """Data pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return C.c_void_p(t.data_ptr())


def tq_pack(codes, bits: int, out=None, stream=None):
    import torch

    n = codes.numel()
    if out is None:
        out = torch.empty((n * bits + 7) // 8, dtype=torch.uint8, device=codes.device)
    _check(lib.tq_pack(_dev(codes, torch.uint8, "codes"), n, bits, _dev(out, torch.uint8, "out"), _stream(stream)), "tq_pack")
    return out


def tq_unpack(src, n: int, bits: int, out=None, stream=None):
    import torch

    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=src.device)
    _check(lib.tq_unpack(_dev(src, torch.uint8, "src"), n, bits, _dev(out, torch.uint8, "out"), _stream(stream)), "tq_unpack")
    return out


class Context:
    """Owner of one tq_ctx (one layer's tables on the current CUDA device)."""

    def __init__(self, layout: int, head_dim: int, num_q_heads: int, num_kv_heads: int, seed: int = 0,
                 centroids=None, signs=None, sketch=None, value_bits=None, key_bits=None, key_format=None):
        self.cfg = tq_config_init(layout, head_dim, num_q_heads, num_kv_heads, seed)
        if value_bits is not None:
            self.cfg.value_bits = value_bits  # main layout: 2 or 4; alternate layout: 2, 3 or 4
        if key_bits is not None:
            self.cfg.key_bits = key_bits  # main layout: 3, 2 or 4; alternate layout: 8, 5, 4, 2 or 16 (fp16 keys)
        if key_format is not None:
            self.cfg.key_format = key_format  # alternate layout, 2-bit keys: TQ_KEY_AFFINE (uint2) or TQ_KEY_SIGNED (int2)
        ptr = C.c_void_p()
        if centroids is None:
            _check(lib.tq_create(C.byref(self.cfg), C.byref(ptr)), "tq_create")
        else:
            c = np.ascontiguousarray(centroids, np.float32)
            s = np.ascontiguousarray(signs, np.float32)
            k = np.ascontiguousarray(sketch, np.float32) if sketch is not None else None
            _check(lib.tq_create_with_tables(C.byref(self.cfg), _np_ptr(c), _np_ptr(s),
                                             _np_ptr(k) if k is not None else None, C.byref(ptr)),
                   "tq_create_with_tables")
        self.ptr = ptr
        self.layout = layout
        self.head_dim = head_dim
        self.num_q_heads = num_q_heads
        self.num_kv_heads = num_kv_heads

    def close(self):
        if getattr(self, "ptr", None) and self.ptr.value:
            lib.tq_destroy(self.ptr)
            self.ptr = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- sizes
    @property
    def bytes_per_token_head(self) -> int:
        return lib.tq_bytes_per_token_head(self.ptr)

    @property
    def page_bytes(self) -> int:
        return lib.tq_page_bytes(self.ptr)

    def workspace_size(self, batch: int, max_ctx: int) -> int:
        n = C.c_size_t()
        _check(lib.tq_workspace_size(self.ptr, batch, max_ctx, C.byref(n)), "tq_workspace_size")
        return n.value

    def set_decode_path(self, path: int):
        """TQ_DECODE_AUTO, TQ_DECODE_MMA_SYNC or TQ_DECODE_TCGEN05 (main layout, head_dim 128)."""
        _check(lib.tq_set_decode_path(self.ptr, path), "tq_set_decode_path")

    def get_tables(self):
        k = 1 << (self.cfg.key_bits - 1 if self.layout == TQ_LAYOUT_MAIN else self.cfg.value_bits)
        d = self.head_dim
        c = np.zeros(k, np.float32)
        b = np.zeros(k - 1, np.float32)
        s = np.zeros(d, np.float32)
        sk = np.zeros((self.cfg.qjl_m, d), np.float32) if self.cfg.qjl_m else None
        _check(lib.tq_get_tables(self.ptr, _np_ptr(c), _np_ptr(b), _np_ptr(s), _np_ptr(sk) if sk is not None else None),
               "tq_get_tables")
        return {"centroids": c, "boundaries": b, "signs": s, "sketch": sk}

    def _check_pool(self, pool):
        if pool is None:
            return
        if pool.dim() != 3 or pool.shape[1] != self.num_kv_heads or pool.shape[2] != self.page_bytes:
            raise ValueError(f"pool must be uint8 [num_blocks, {self.num_kv_heads}, {self.page_bytes}]")

    def _check_bt(self, bt, batch):
        if bt.dim() != 2 or bt.shape[0] != batch:
            raise ValueError("block_table must be int32 [batch, max_blocks]")

    # -- write path
    def encode_flush(self, k, v, start_pos, block_table, pool, n_tokens=None, stream=None):
        """k, v: fp16 [B, Hkv, src_tokens, d]; start_pos int32 [B]; block_table int32 [B, max_blocks]."""
        import torch

        bsz, hkv, src, d = k.shape
        n = src if n_tokens is None else n_tokens
        if v.shape != k.shape or hkv != self.num_kv_heads or d != self.head_dim or start_pos.numel() != bsz:
            raise ValueError("k, v must be [batch, Hkv, src_tokens, d] and start_pos [batch]")
        self._check_pool(pool)
        self._check_bt(block_table, bsz)
        _check(lib.tq_encode_flush(self.ptr, _dev(k, torch.float16, "k"), _dev(v, torch.float16, "v"), bsz, src, n,
                                   _dev(start_pos, torch.int32, "start_pos"), _dev(block_table, torch.int32, "block_table"),
                                   block_table.shape[1], _dev(pool, torch.uint8, "pool"), pool.shape[0], _stream(stream)),
               "tq_encode_flush")

    def append_token(self, k_new, v_new, pos, ring_k, ring_v, block_table, pool, stream=None):
        import torch

        bsz = k_new.shape[0]
        if tuple(k_new.shape) != (bsz, self.num_kv_heads, self.head_dim) or v_new.shape != k_new.shape:
            raise ValueError("k_new, v_new must be [batch, Hkv, d]")
        if tuple(ring_k.shape) != (bsz, self.num_kv_heads, 128, self.head_dim) or ring_v.shape != ring_k.shape:
            raise ValueError("ring_k, ring_v must be [batch, Hkv, 128, d]")
        if pos.numel() != bsz:
            raise ValueError("pos must be [batch]")
        self._check_pool(pool)
        self._check_bt(block_table, bsz)
        _check(lib.tq_append_token(self.ptr, _dev(k_new, torch.float16, "k_new"), _dev(v_new, torch.float16, "v_new"),
                                   _dev(pos, torch.int32, "pos"), k_new.shape[0], _dev(ring_k, torch.float16, "ring_k"),
                                   _dev(ring_v, torch.float16, "ring_v"), _dev(block_table, torch.int32, "block_table"),
                                   block_table.shape[1], _dev(pool, torch.uint8, "pool"), pool.shape[0], _stream(stream)),
               "tq_append_token")

    # -- read path
    def decode_attention(self, q, pool, block_table, n_compressed, ring_k, ring_v, n_buf, max_ctx, out, workspace,
                         stream=None):
        import torch

        bsz = q.shape[0]
        if tuple(q.shape) != (bsz, self.num_q_heads, self.head_dim) or tuple(out.shape) != tuple(q.shape):
            raise ValueError("q must be [batch, Hq, d] fp16 and out [batch, Hq, d] fp32")
        if n_compressed.numel() != bsz or (n_buf is not None and n_buf.numel() != bsz):
            raise ValueError("n_compressed / n_buf must be [batch]")
        if ring_k is not None and (tuple(ring_k.shape) != (bsz, self.num_kv_heads, 128, self.head_dim)
                                   or ring_v is None or ring_v.shape != ring_k.shape):
            raise ValueError("ring_k, ring_v must be [batch, Hkv, 128, d]")
        self._check_pool(pool)
        self._check_bt(block_table, bsz)
        _check(lib.tq_decode_attention(self.ptr, _dev(q, torch.float16, "q"), q.shape[0],
                                       _dev(pool, torch.uint8, "pool") if pool is not None else None,
                                       pool.shape[0] if pool is not None else 0,
                                       _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
                                       _dev(n_compressed, torch.int32, "n_compressed"),
                                       _dev(ring_k, torch.float16, "ring_k"), _dev(ring_v, torch.float16, "ring_v"),
                                       _dev(n_buf, torch.int32, "n_buf"), max_ctx, _dev(out, torch.float32, "out"),
                                       _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)),
               "tq_decode_attention")

    def decode_attention_static(self, q, pool, block_table, n_compressed, ring_k, ring_v, n_buf, max_ctx, out,
                                stream=None):
        """tq_decode_attention_static: as decode_attention, scratch in the library's fixed device array."""
        import torch

        bsz = q.shape[0]
        if tuple(q.shape) != (bsz, self.num_q_heads, self.head_dim) or tuple(out.shape) != tuple(q.shape):
            raise ValueError("q must be [batch, Hq, d] fp16 and out [batch, Hq, d] fp32")
        self._check_pool(pool)
        self._check_bt(block_table, bsz)
        _check(lib.tq_decode_attention_static(self.ptr, _dev(q, torch.float16, "q"), bsz,
                                              _dev(pool, torch.uint8, "pool") if pool is not None else None,
                                              pool.shape[0] if pool is not None else 0,
                                              _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
                                              _dev(n_compressed, torch.int32, "n_compressed"),
                                              _dev(ring_k, torch.float16, "ring_k"), _dev(ring_v, torch.float16, "ring_v"),
                                              _dev(n_buf, torch.int32, "n_buf"), max_ctx,
                                              _dev(out, torch.float32, "out"), _stream(stream)),
               "tq_decode_attention_static")

    def dequantize(self, pool, block_table, n_compressed, k_out, v_out, ring_k=None, ring_v=None, n_buf=None,
                   stream=None):
        """tq_dequantize (fp16 k_out / v_out) or tq_dequantize_bf16 (bf16 k_out / v_out): rows
        0..n_compressed[b]-1 of k_out / v_out [batch, Hkv, max_tokens, d] from the pool, followed by the
        n_buf[b] ring tokens when a ring is given."""
        import torch

        bsz = k_out.shape[0]
        shape = (bsz, self.num_kv_heads, k_out.shape[2], self.head_dim)
        if tuple(k_out.shape) != shape or tuple(v_out.shape) != shape:
            raise ValueError("k_out and v_out must be [batch, Hkv, max_tokens, d]")
        if k_out.dtype not in (torch.float16, torch.bfloat16) or v_out.dtype != k_out.dtype:
            raise ValueError("k_out and v_out must both be fp16 or both bf16")
        fn, name = ((lib.tq_dequantize_bf16, "tq_dequantize_bf16") if k_out.dtype == torch.bfloat16
                    else (lib.tq_dequantize, "tq_dequantize"))
        self._check_pool(pool)
        self._check_bt(block_table, bsz)
        _check(fn(self.ptr, _dev(pool, torch.uint8, "pool"), pool.shape[0],
                  _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
                  _dev(n_compressed, torch.int32, "n_compressed"),
                  _dev(ring_k, torch.float16, "ring_k"), _dev(ring_v, torch.float16, "ring_v"),
                  _dev(n_buf, torch.int32, "n_buf"), bsz, k_out.shape[2],
                  _dev(k_out, k_out.dtype, "k_out"), _dev(v_out, v_out.dtype, "v_out"),
                  _stream(stream)), name)

    # -- diagnostics
    def device_errors(self, stream=None) -> int:
        f = C.c_uint32()
        _check(lib.tq_get_device_errors(self.ptr, C.byref(f), _stream(stream)), "tq_get_device_errors")
        return f.value

    @property
    def launch_count(self) -> int:
        return lib.tq_launch_count(self.ptr)

    def profile_begin(self):
        _check(lib.tq_profile_begin(self.ptr), "tq_profile_begin")

    def profile_end(self) -> dict:
        p = tq_profile()
        _check(lib.tq_profile_end(self.ptr, C.byref(p)), "tq_profile_end")
        r = {f: getattr(p, f) for f, _ in tq_profile._fields_}
        r["decode_kernel"] = r["decode_kernel"].decode() if r["decode_kernel"] else None
        return r
