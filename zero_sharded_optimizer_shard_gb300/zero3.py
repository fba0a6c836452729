"""ctypes binding of the C ABI in include/zero3.h.

Argument marshalling only: every function forwards to the entry point of the
same name in libzero3.so, and every step of the computation runs in the CUDA
library.  Device pointers are plain integers (e.g. ``tensor.data_ptr()``);
streams are ``cudaStream_t`` handles as integers (e.g.
``torch.cuda.current_stream().cuda_stream``), 0 for the legacy default stream.
A non-OK status raises ``Zero3Error``.  If the library has not been built the
import of any compute function raises: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

from .build import lib_path

OK, EINVAL, ESTATE, ECUDA, ENOMEM, EIO = 0, 1, 2, 3, 4, 5
BF16, F32 = 0, 1
NOT_AVAILABLE, INFLIGHT, AVAILABLE = 0, 1, 2
MAX_RANKS = 64

_c_i64_p = C.POINTER(C.c_int64)
_c_i32_p = C.POINTER(C.c_int32)
_vp = C.c_void_p


class AdamWHparams(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double)]


class PlanInfo(C.Structure):
    _fields_ = [("n_ranks", C.c_int32), ("n_submodules", C.c_int32),
                ("n_tensors", C.c_int64), ("n_partitioned", C.c_int64),
                ("n_persistent", C.c_int64), ("psi_p", C.c_int64), ("psi_pad", C.c_int64),
                ("shard_len", C.c_int64), ("psi_s", C.c_int64),
                ("persistence_threshold", C.c_int64), ("reduce_bucket_size", C.c_int64),
                ("n_buckets", C.c_int64)]


class TensorInfo(C.Structure):
    _fields_ = [("numel", C.c_int64), ("offset", C.c_int64), ("persistent", C.c_int32),
                ("submodule", C.c_int32), ("first_rank", C.c_int32), ("last_rank", C.c_int32),
                ("n_segments", C.c_int64)]


class Segment(C.Structure):
    _fields_ = [("rank", C.c_int32), ("reserved", C.c_int32), ("shard_off", C.c_int64),
                ("tensor_off", C.c_int64), ("len", C.c_int64)]


class PersistState(C.Structure):
    _fields_ = [("grads", C.POINTER(_vp)), ("master", _vp), ("m", _vp), ("v", _vp),
                ("param", _vp)]


class PrefetchConfig(C.Structure):
    _fields_ = [("prefetch_bucket_size", C.c_int64), ("max_live_parameters", C.c_int64),
                ("max_reuse_distance", C.c_int64)]


class CoordinatorStats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("steps", "gathers", "prefetched", "prefetch_hits",
                                          "reuse_hits", "evictions", "trace_misses",
                                          "gathered_elems", "peak_live_elems", "live_elems",
                                          "gather_calls", "gather_launches", "compute_waits")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class Zero3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_LIB: Optional[C.CDLL] = None

# (name, restype, argtypes)
_SIGS = [
    ("zero3_partition", C.c_int, [_c_i64_p, _c_i32_p, C.c_int64, C.c_int32, C.c_int64, C.c_int64,
                                  C.POINTER(_vp)]),
    ("zero3_plan_info_get", C.c_int, [_vp, C.POINTER(PlanInfo)]),
    ("zero3_plan_tensor", C.c_int, [_vp, C.c_int64, C.POINTER(TensorInfo)]),
    ("zero3_plan_segments", C.c_int, [_vp, C.c_int64, C.POINTER(Segment), C.c_int64, _c_i64_p]),
    ("zero3_plan_bucket", C.c_int, [_vp, C.c_int64, _c_i64_p, _c_i64_p]),
    ("zero3_plan_submodule", C.c_int, [_vp, C.c_int32, _c_i64_p, _c_i64_p]),
    ("zero3_plan_destroy", None, [_vp]),
    ("zero3_reduce_scatter", C.c_int, [_vp, C.POINTER(_vp), C.c_int64, C.c_int64, C.c_int64,
                                       C.POINTER(_vp), C.c_int, _vp]),
    ("zero3_adamw_step", C.c_int, [_vp, C.POINTER(AdamWHparams), C.c_int64, C.POINTER(_vp),
                                   C.c_int, C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp),
                                   C.POINTER(_vp), C.c_int64, C.c_int64, _vp]),
    ("zero3_allgather", C.c_int, [_vp, C.POINTER(_vp), _vp, C.c_int64, C.c_int64, _vp]),
    ("zero3_step", C.c_int, [_vp, C.POINTER(AdamWHparams), C.c_int64, C.POINTER(_vp), C.c_int64,
                             C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp), _vp,
                             C.POINTER(PersistState), C.c_int64, C.c_int64, _vp]),
    ("zero3_step_stage12", C.c_int, [_vp, C.POINTER(AdamWHparams), C.c_int64, C.POINTER(_vp),
                                     C.c_int64, C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp),
                                     C.POINTER(_vp), C.c_int64, C.c_int64, _vp]),
    ("zero3_step_qwz", C.c_int, [_vp, C.POINTER(AdamWHparams), C.c_int64, C.POINTER(_vp),
                                 C.c_int64, C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp),
                                 C.POINTER(_vp), C.c_int32, C.POINTER(_vp), C.POINTER(_vp),
                                 C.POINTER(PersistState), C.c_int64, C.c_int64, _vp]),
    ("zero3_quantize_shards", C.c_int, [_vp, C.POINTER(_vp), C.c_int32, C.POINTER(_vp),
                                        C.POINTER(_vp), C.c_int64, C.c_int64, _vp]),
    ("zero3_allgather_qwz", C.c_int, [_vp, C.c_int32, C.POINTER(_vp), C.POINTER(_vp), _vp,
                                      C.c_int64, C.c_int64, _vp]),
    ("zero3_persistent_step", C.c_int, [_vp, C.POINTER(AdamWHparams), C.c_int64,
                                        C.POINTER(PersistState), _vp]),
    ("zero3_cast_params", C.c_int, [_vp, C.POINTER(_vp), C.POINTER(_vp), _vp,
                                    C.POINTER(PersistState), C.c_int64, C.c_int64, _vp]),
    ("zero3_fetch_submodule", C.c_int, [_vp, C.c_int32, C.POINTER(_vp), _vp, _vp, _vp]),
    ("zero3_fetch_submodules", C.c_int, [_vp, _c_i32_p, C.c_int32, C.POINTER(_vp), _vp,
                                         C.POINTER(_vp), _vp]),
    ("zero3_release_submodule", C.c_int, [_vp, C.c_int32]),
    ("zero3_submodule_status", C.c_int, [_vp, C.c_int32, _c_i32_p]),
    ("zero3_submodule_wait", C.c_int, [_vp, C.c_int32]),
    ("zero3_coordinator_create", C.c_int, [_vp, _c_i32_p, C.c_int64, C.POINTER(_vp), _vp, _vp,
                                           C.c_int64, C.POINTER(PrefetchConfig), _vp, _vp,
                                           C.POINTER(_vp)]),
    ("zero3_coordinator_fetch", C.c_int, [_vp, C.c_int32, C.POINTER(_vp)]),
    ("zero3_coordinator_release", C.c_int, [_vp, C.c_int32]),
    ("zero3_coordinator_status", C.c_int, [_vp, C.c_int32, _c_i32_p]),
    ("zero3_coordinator_next_step", C.c_int, [_vp]),
    ("zero3_coordinator_get_stats", C.c_int, [_vp, C.POINTER(CoordinatorStats)]),
    ("zero3_coordinator_destroy", None, [_vp]),
    ("zero3_save_shard", C.c_int, [_vp, C.c_int32, C.c_int64, _vp, _vp, _vp, C.c_char_p, _vp]),
    ("zero3_load_shard", C.c_int, [_vp, C.c_int32, _c_i64_p, _vp, _vp, _vp, C.c_char_p, _vp]),
    ("zero3_save_persistent", C.c_int, [_vp, C.c_int64, C.POINTER(PersistState), C.c_char_p, _vp]),
    ("zero3_load_persistent", C.c_int, [_vp, _c_i64_p, C.POINTER(PersistState), C.c_char_p, _vp]),
    ("zero3_save_16bit_weights", C.c_int, [_vp, _vp, _vp, C.c_char_p, _vp]),
    ("zero3_merge_shards", C.c_int, [_vp, C.POINTER(C.c_char_p), C.c_char_p, C.c_char_p]),
    ("zero3_plan_memory_bytes", C.c_int, [_vp, C.c_int32, C.POINTER(C.c_double)]),
    ("zero3_memory_bytes", C.c_int, [C.c_int32, C.c_double, C.c_int32, C.POINTER(C.c_double)]),
    ("zero3_comm_elems", C.c_int, [C.c_int32, C.c_double, C.c_int32, C.POINTER(C.c_double)]),
    ("zero3_sync", C.c_int, [_vp]),
    ("zero3_status_string", C.c_char_p, [C.c_int]),
]

EXPORTED = [s[0] for s in _SIGS]


def load() -> C.CDLL:
    """Loads libzero3.so from the package directory (raises if missing)."""
    global _LIB
    if _LIB is None:
        path = lib_path("libzero3.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "zero_sharded_optimizer_shard_gb300.build.build_all()")
        lib = C.CDLL(path)
        for name, res, args in _SIGS:
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _LIB = lib
    return _LIB


def status_string(s: int) -> str:
    return load().zero3_status_string(s).decode()


def _check(st: int, where: str) -> None:
    if st != OK:
        raise Zero3Error(st, where)


def _ptrs(seq: Optional[Sequence[Optional[int]]]):
    if seq is None:
        return None
    arr = (_vp * len(seq))(*[(p or None) for p in seq])
    return arr


def hparams(lr=5e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01) -> AdamWHparams:
    return AdamWHparams(lr, beta1, beta2, eps, weight_decay)


class Plan:
    """Owner of a zero3_plan* (destroyed with the object)."""

    def __init__(self, numels: Sequence[int], submodule_of: Optional[Sequence[int]],
                 n_ranks: int, threshold: int = 100_000, bucket: int = 500_000_000):
        lib = load()
        n = len(numels)
        nb = (C.c_int64 * max(n, 1))(*numels)
        sb = (C.c_int32 * max(n, 1))(*submodule_of) if submodule_of is not None else None
        out = _vp()
        _check(lib.zero3_partition(nb, sb, n, n_ranks, threshold, bucket, C.byref(out)),
               "zero3_partition")
        self.handle = out
        self._lib = lib
        info = PlanInfo()
        _check(lib.zero3_plan_info_get(out, C.byref(info)), "zero3_plan_info_get")
        self.info = info

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            self._lib.zero3_plan_destroy(h)
            self.handle = None

    # --- queries
    def tensor(self, t: int) -> TensorInfo:
        ti = TensorInfo()
        _check(self._lib.zero3_plan_tensor(self.handle, t, C.byref(ti)), "zero3_plan_tensor")
        return ti

    def segments(self, t: int):
        n = C.c_int64()
        _check(self._lib.zero3_plan_segments(self.handle, t, None, 0, C.byref(n)),
               "zero3_plan_segments")
        arr = (Segment * max(n.value, 1))()
        _check(self._lib.zero3_plan_segments(self.handle, t, arr, n.value, C.byref(n)),
               "zero3_plan_segments")
        return [(s.rank, s.shard_off, s.tensor_off, s.len) for s in arr[:n.value]]

    def bucket(self, b: int):
        lo, hi = C.c_int64(), C.c_int64()
        _check(self._lib.zero3_plan_bucket(self.handle, b, C.byref(lo), C.byref(hi)),
               "zero3_plan_bucket")
        return lo.value, hi.value

    def submodule(self, k: int):
        nt, ne = C.c_int64(), C.c_int64()
        _check(self._lib.zero3_plan_submodule(self.handle, k, C.byref(nt), C.byref(ne)),
               "zero3_plan_submodule")
        return nt.value, ne.value


def persist_state(grads: Sequence[int], master: int, m: int, v: int, param: int):
    g = _ptrs(grads)
    ps = PersistState(C.cast(g, C.POINTER(_vp)), master, m, v, param)
    ps._keep = g  # keep the pointer array alive with the struct
    return ps


def _ps_ref(ps):
    return C.byref(ps) if ps is not None else None


def zero3_reduce_scatter(plan: Plan, grads, grads_origin, flat_lo, flat_hi, shard_grad,
                         out_dtype=F32, stream=0):
    _check(plan._lib.zero3_reduce_scatter(plan.handle, _ptrs(grads), grads_origin, flat_lo,
                                          flat_hi, _ptrs(shard_grad), out_dtype, stream),
           "zero3_reduce_scatter")


def zero3_adamw_step(plan: Plan, hp, t, shard_grad, grad_dtype, master, m, v, sparam,
                     flat_lo, flat_hi, stream=0):
    _check(plan._lib.zero3_adamw_step(plan.handle, C.byref(hp), t, _ptrs(shard_grad), grad_dtype,
                                      _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(sparam), flat_lo,
                                      flat_hi, stream), "zero3_adamw_step")


def zero3_allgather(plan: Plan, sparam, full, flat_lo, flat_hi, stream=0):
    _check(plan._lib.zero3_allgather(plan.handle, _ptrs(sparam), full, flat_lo, flat_hi, stream),
           "zero3_allgather")


def zero3_step(plan: Plan, hp, t, grads, grads_origin, master, m, v, sparam, full, persist,
               flat_lo, flat_hi, stream=0):
    _check(plan._lib.zero3_step(plan.handle, C.byref(hp), t, _ptrs(grads), grads_origin,
                                _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(sparam), full,
                                _ps_ref(persist), flat_lo, flat_hi, stream), "zero3_step")


def zero3_step_stage12(plan: Plan, hp, t, grads, grads_origin, master, m, v, params, flat_lo,
                       flat_hi, stream=0):
    _check(plan._lib.zero3_step_stage12(plan.handle, C.byref(hp), t, _ptrs(grads), grads_origin,
                                        _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(params), flat_lo,
                                        flat_hi, stream), "zero3_step_stage12")


QWZ_BLOCK = 256


def zero3_step_qwz(plan: Plan, hp, t, grads, grads_origin, master, m, v, sparam, codes, scales,
                   persist, flat_lo, flat_hi, stream=0, bits=8):
    _check(plan._lib.zero3_step_qwz(plan.handle, C.byref(hp), t, _ptrs(grads), grads_origin,
                                    _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(sparam), bits,
                                    _ptrs(codes), _ptrs(scales), _ps_ref(persist), flat_lo,
                                    flat_hi, stream), "zero3_step_qwz")


def zero3_quantize_shards(plan: Plan, sparam, codes, scales, flat_lo, flat_hi, stream=0, bits=8):
    _check(plan._lib.zero3_quantize_shards(plan.handle, _ptrs(sparam), bits, _ptrs(codes),
                                           _ptrs(scales), flat_lo, flat_hi, stream),
           "zero3_quantize_shards")


def zero3_allgather_qwz(plan: Plan, codes, scales, full, flat_lo, flat_hi, stream=0, bits=8):
    _check(plan._lib.zero3_allgather_qwz(plan.handle, bits, _ptrs(codes), _ptrs(scales), full,
                                         flat_lo, flat_hi, stream), "zero3_allgather_qwz")


def zero3_persistent_step(plan: Plan, hp, t, persist, stream=0):
    _check(plan._lib.zero3_persistent_step(plan.handle, C.byref(hp), t, _ps_ref(persist), stream),
           "zero3_persistent_step")


def zero3_cast_params(plan: Plan, master, sparam, full, persist, flat_lo, flat_hi, stream=0):
    _check(plan._lib.zero3_cast_params(plan.handle, _ptrs(master), _ptrs(sparam), full or None,
                                       _ps_ref(persist), flat_lo, flat_hi, stream),
           "zero3_cast_params")


def zero3_fetch_submodule(plan: Plan, k, sparam, persist_param, out, stream=0):
    _check(plan._lib.zero3_fetch_submodule(plan.handle, k, _ptrs(sparam), persist_param or None,
                                           out or None, stream), "zero3_fetch_submodule")


def zero3_fetch_submodules(plan: Plan, ks, sparam, persist_param, outs, stream=0):
    ka = (C.c_int32 * max(len(ks), 1))(*ks)
    _check(plan._lib.zero3_fetch_submodules(plan.handle, ka, len(ks), _ptrs(sparam),
                                            persist_param or None, _ptrs(outs), stream),
           "zero3_fetch_submodules")


def zero3_release_submodule(plan: Plan, k):
    _check(plan._lib.zero3_release_submodule(plan.handle, k), "zero3_release_submodule")


def zero3_submodule_status(plan: Plan, k) -> int:
    s = C.c_int32()
    _check(plan._lib.zero3_submodule_status(plan.handle, k, C.byref(s)), "zero3_submodule_status")
    return s.value


def zero3_submodule_wait(plan: Plan, k):
    _check(plan._lib.zero3_submodule_wait(plan.handle, k), "zero3_submodule_wait")


class Coordinator:
    """Owner of a zero3_coordinator* (prefetching gathers into an arena)."""

    def __init__(self, plan: Plan, trace, sparam, persist_param, arena, arena_elems,
                 prefetch_bucket_size=500_000_000, max_live_parameters=1_000_000_000,
                 max_reuse_distance=1_000_000_000, compute_stream=0, prefetch_stream=0):
        lib = plan._lib
        self._lib = lib
        self.plan = plan  # keeps the plan alive
        tr = list(trace or [])
        ta = (C.c_int32 * max(len(tr), 1))(*tr)
        self.cfg = PrefetchConfig(prefetch_bucket_size, max_live_parameters, max_reuse_distance)
        out = _vp()
        _check(lib.zero3_coordinator_create(plan.handle, ta if tr else None, len(tr),
                                            _ptrs(sparam), persist_param or None, arena or None,
                                            arena_elems, C.byref(self.cfg), compute_stream,
                                            prefetch_stream, C.byref(out)),
               "zero3_coordinator_create")
        self.handle = out

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            self._lib.zero3_coordinator_destroy(h)
            self.handle = None

    def fetch(self, k: int) -> int:
        p = _vp()
        _check(self._lib.zero3_coordinator_fetch(self.handle, k, C.byref(p)),
               "zero3_coordinator_fetch")
        return p.value or 0

    def release(self, k: int) -> None:
        _check(self._lib.zero3_coordinator_release(self.handle, k), "zero3_coordinator_release")

    def status(self, k: int) -> int:
        s = C.c_int32()
        _check(self._lib.zero3_coordinator_status(self.handle, k, C.byref(s)),
               "zero3_coordinator_status")
        return s.value

    def next_step(self) -> None:
        _check(self._lib.zero3_coordinator_next_step(self.handle), "zero3_coordinator_next_step")

    def stats(self) -> dict:
        st = CoordinatorStats()
        _check(self._lib.zero3_coordinator_get_stats(self.handle, C.byref(st)),
               "zero3_coordinator_get_stats")
        return st.as_dict()


def _path(path) -> bytes:
    return os.fsencode(path)


def zero3_save_shard(plan: Plan, rank, t, master, m, v, path, stream=0):
    _check(plan._lib.zero3_save_shard(plan.handle, rank, t, master, m, v, _path(path), stream),
           "zero3_save_shard")


def zero3_load_shard(plan: Plan, rank, master, m, v, path, stream=0) -> int:
    t = C.c_int64()
    _check(plan._lib.zero3_load_shard(plan.handle, rank, C.byref(t), master, m, v, _path(path),
                                      stream), "zero3_load_shard")
    return t.value


def zero3_save_persistent(plan: Plan, t, persist, path, stream=0):
    _check(plan._lib.zero3_save_persistent(plan.handle, t, _ps_ref(persist), _path(path), stream),
           "zero3_save_persistent")


def zero3_load_persistent(plan: Plan, persist, path, stream=0) -> int:
    t = C.c_int64()
    _check(plan._lib.zero3_load_persistent(plan.handle, C.byref(t), _ps_ref(persist), _path(path),
                                           stream), "zero3_load_persistent")
    return t.value


def zero3_save_16bit_weights(plan: Plan, full, persist_param, path, stream=0):
    _check(plan._lib.zero3_save_16bit_weights(plan.handle, full or None, persist_param or None,
                                              _path(path), stream), "zero3_save_16bit_weights")


def zero3_merge_shards(plan: Plan, shard_paths, persistent_path, out_path):
    arr = (C.c_char_p * len(shard_paths))(*[_path(x) for x in shard_paths])
    _check(plan._lib.zero3_merge_shards(plan.handle, arr,
                                        _path(persistent_path) if persistent_path else None,
                                        _path(out_path)), "zero3_merge_shards")


def zero3_plan_memory_bytes(plan: Plan, stage) -> float:
    out = C.c_double()
    _check(plan._lib.zero3_plan_memory_bytes(plan.handle, stage, C.byref(out)),
           "zero3_plan_memory_bytes")
    return out.value


def zero3_memory_bytes(stage, psi, n_d) -> float:
    out = C.c_double()
    _check(load().zero3_memory_bytes(stage, psi, n_d, C.byref(out)), "zero3_memory_bytes")
    return out.value


def zero3_comm_elems(stage, psi, n_d) -> float:
    out = C.c_double()
    _check(load().zero3_comm_elems(stage, psi, n_d, C.byref(out)), "zero3_comm_elems")
    return out.value


def zero3_sync(stream=0):
    _check(load().zero3_sync(stream), "zero3_sync")


def raw_status(fn_name: str, *args) -> int:
    """Calls an entry point and returns its status without raising (tests of
    the error paths)."""
    return getattr(load(), fn_name)(*args)
