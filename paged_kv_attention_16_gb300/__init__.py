"""Unified paged attention over a continuous batch, for GB300 (sm_103a).

The compute lives in a C-ABI CUDA library (libpa.so, header include/pa.h);
`paged_kv_attention_16_gb300.pa` is the thin ctypes binding over it.  The
binding is imported lazily so that the seeded input generators
(`paged_kv_attention_16_gb300.inputs`) can be used without a GPU.
"""
import importlib

__all__ = ["pa", "inputs", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
