"""ctypes binding of libzero3_synth.so, the device side of the seeded
generator defined in synth.py (same definition, written independently in
CUDA).  Input plumbing only."""
from __future__ import annotations

import ctypes as C
import os

from .build import lib_path

_LIB = None


def load() -> C.CDLL:
    global _LIB
    if _LIB is None:
        path = lib_path("libzero3_synth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run build.build_all()")
        lib = C.CDLL(path)
        lib.zero3synth_normal.restype = C.c_int
        lib.zero3synth_normal.argtypes = [C.c_uint64, C.c_int64, C.c_int64, C.c_int64, C.c_int64,
                                          C.c_int64, C.c_double, C.c_double, C.c_double,
                                          C.c_int32, C.c_void_p, C.c_void_p]
        _LIB = lib
    return _LIB


def normal(out_ptr: int, n: int, *, seed: int, stream_id: int, step: int, rank: int,
           index0: int, sigma: float, outlier_p: float = 0.0, outlier_sigma: float = 0.0,
           bf16: bool = True, cuda_stream: int = 0) -> None:
    """Writes samples for flat indices index0 .. index0+n-1 to out_ptr."""
    err = load().zero3synth_normal(seed, stream_id, step, rank, index0, n, sigma, outlier_p,
                                   outlier_sigma, 1 if bf16 else 0, out_ptr, cuda_stream)
    if err != 0:
        raise RuntimeError(f"zero3synth_normal failed with cudaError {err}")
