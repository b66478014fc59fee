"""TurboQuant-style compressed KV cache and decode attention for NVIDIA GB300.

The compute lives in ``libtq.so`` (hand-written CUDA for sm_103a behind the
C ABI of ``include/tq.h``); this package holds the sources (``csrc/``), the
in-place build (``build.py``) and a ctypes binding with the same names as the
C entry points (``binding.py``).  The binding is imported on first use of any
of its names, so ``kv_cache_quantization_tq_gb300.build`` works before the
library exists; using the binding without a built library raises ImportError.
"""
_EXPORTS = (
    "TQ_DECODE_AUTO",
    "TQ_DECODE_MMA_SYNC",
    "TQ_DECODE_TCGEN05",
    "TQ_KEY_AFFINE",
    "TQ_KEY_SIGNED",
    "TQ_LAYOUT_ALT",
    "TQ_LAYOUT_MAIN",
    "Context",
    "TQError",
    "lib",
    "tq_config_init",
    "tq_generate_tables",
    "tq_lloyd_max",
    "tq_pack",
    "tq_pack_host",
    "tq_should_materialize",
    "tq_unpack",
    "tq_unpack_host",
)
__all__ = list(_EXPORTS) + ["binding", "build"]


def __getattr__(name):
    if name in _EXPORTS or name == "binding":
        import importlib

        mod = importlib.import_module(__name__ + ".binding")
        return mod if name == "binding" else getattr(mod, name)
    raise AttributeError(name)
