"""TurboQuant-style compressed KV cache and decode attention for NVIDIA GB300.

The compute lives in ``libtq.so`` (hand-written CUDA for sm_103a behind the
C ABI of ``include/tq.h``); this package holds the sources (``csrc/``), the
in-place build (``build.py``) and a ctypes binding with the same names as the
C entry points (``binding.py``).
"""
from .binding import (  # noqa: F401
    TQ_LAYOUT_ALT,
    TQ_LAYOUT_MAIN,
    Context,
    TQError,
    lib,
    tq_config_init,
    tq_generate_tables,
    tq_lloyd_max,
    tq_pack,
    tq_pack_host,
    tq_unpack,
    tq_unpack_host,
)
