"""ZeRO-3 sharded mixed-precision AdamW hot path for GB300 (sm_103a).

The compute lives in the C-ABI library ``libzero3.so`` (CUDA kernels plus a
host planner); ``zero3`` is its thin ctypes binding.  Submodules load lazily so
that the shape lists (``workloads``) and the seeded generator (``synth``) can
be imported on machines without a GPU or without the built library.
"""
__all__ = ["zero3", "workloads", "synth", "build"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
