"""Unified paged attention over a continuous batch, for GB300 (sm_103a).

The compute lives in a C-ABI CUDA library (libpa.so, header include/pa.h);
`paged_kv_attention_16_gb300.pa` is the thin ctypes binding over it.  The
binding is imported lazily so that the seeded input generators
(`paged_kv_attention_16_gb300.inputs`) can be used without a GPU.
"""

__all__ = ["pa", "inputs"]


def __getattr__(name):
    if name == "pa":
        from . import pa as _pa
        return _pa
    if name == "inputs":
        from . import inputs as _inputs
        return _inputs
    raise AttributeError(name)
