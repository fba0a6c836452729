"""Host-side tests of the C ABI: exports, planner parity with the oracle,
accounting, argument validation and the submodule state machine's host
transitions.  No call here launches a kernel: every compute call below
carries at least one invalid argument, which the library rejects before it
touches the GPU."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle as O
from zero_sharded_optimizer_shard_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zero3.h")


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zero3_[a-z0-9_]+)\s*\(", src)))


def test_header_lists_every_binding_function():
    from zero_sharded_optimizer_shard_gb300 import zero3
    assert header_functions() == sorted(zero3.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_synth_library_exports(lib):
    from zero_sharded_optimizer_shard_gb300 import synth_device
    assert hasattr(synth_device.load(), "zero3synth_normal")


# ---------------------------------------------------------------- planner parity
def _compare_plan(numels, subs, nd, thr, bucket):
    from zero_sharded_optimizer_shard_gb300 import zero3
    ref = O.partition(numels, subs, nd, thr, bucket)
    p = zero3.Plan(numels, subs, nd, thr, bucket)
    i = p.info
    assert (i.n_ranks, i.psi_p, i.psi_pad, i.shard_len, i.psi_s) == \
        (nd, ref.psi_p, ref.psi_pad, ref.shard_len, ref.psi_s)
    assert i.n_tensors == len(numels)
    assert i.n_persistent == sum(ref.persistent)
    assert i.n_buckets == len(ref.buckets)
    assert [p.bucket(b) for b in range(i.n_buckets)] == ref.buckets
    assert i.n_submodules == ref.n_submodules
    for k in range(i.n_submodules):
        assert p.submodule(k) == (len(ref.submodules.get(k, [])), ref.submodule_numel(k))
    for t in range(len(numels)):
        ti = p.tensor(t)
        assert (ti.numel, ti.offset, bool(ti.persistent), ti.submodule) == \
            (ref.numel[t], ref.offset[t], ref.persistent[t], ref.submodule[t])
        segs = p.segments(t)
        assert segs == ref.segments[t]
        if segs:
            assert (ti.first_rank, ti.last_rank) == (segs[0][0], segs[-1][0])
        else:
            assert (ti.first_rank, ti.last_rank) == (-1, -1)


@pytest.mark.parametrize("name", ["toy_mlp", "gpt2_small", "decoder_1p3b", "llama_7b_rank0",
                                  "ragged"])
def test_planner_matches_oracle_on_workloads(lib, name):
    w = W.BY_NAME[name]()
    _compare_plan(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)


def test_planner_matches_oracle_brute_force(lib):
    rng = np.random.default_rng(7)
    for trial in range(400):
        nd = int(rng.integers(1, 10))
        n_t = int(rng.integers(0, 9))
        numels = [int(x) for x in rng.integers(0, 40, n_t)]
        subs = [int(x) for x in rng.integers(0, 4, n_t)] if rng.random() < 0.5 else None
        _compare_plan(numels, subs, nd, int(rng.integers(0, 20)), int(rng.integers(1, 30)))


def test_planner_large_rank_counts(lib):
    _compare_plan([10**6 + 3, 5, 77777, 2 * 10**5], None, 64, 100_000, 10**5)
    _compare_plan([1], None, 64, 0, 1)


# ---------------------------------------------------------------- accounting
def test_accounting_matches_oracle(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    for stage in range(4):
        for psi, nd in [(7e9, 4), (7.5e9, 64), (1.3e9, 8), (1.0, 1)]:
            assert zero3.zero3_memory_bytes(stage, psi, nd) == pytest.approx(
                O.memory_bytes(stage, psi, nd), rel=1e-15)
            assert 2 * zero3.zero3_comm_elems(stage, psi, nd) == pytest.approx(
                O.ring_send_bytes(stage, psi, nd), rel=1e-15)
    # the pages' 7B / 4 GPU numbers through the library
    assert zero3.zero3_memory_bytes(3, 7e9, 4) == 28e9
    assert 2 * zero3.zero3_comm_elems(3, 7e9, 4) == pytest.approx(31.5e9)


def test_accounting_rejects_bad_arguments(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    out = C.c_double()
    assert zero3.raw_status("zero3_memory_bytes", 4, 1.0, 4, C.byref(out)) == zero3.EINVAL
    assert zero3.raw_status("zero3_memory_bytes", 3, 1.0, 0, C.byref(out)) == zero3.EINVAL
    assert zero3.raw_status("zero3_comm_elems", -1, 1.0, 4, C.byref(out)) == zero3.EINVAL
    assert zero3.raw_status("zero3_comm_elems", 3, 1.0, 4, None) == zero3.EINVAL


# ---------------------------------------------------------------- validation
def test_partition_rejects_bad_arguments(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    out = C.c_void_p()
    n = (C.c_int64 * 2)(10, 20)
    neg = (C.c_int64 * 2)(10, -1)
    bad_sub = (C.c_int32 * 2)(0, -3)
    for args in [(n, None, 2, 0, 0, 1), (n, None, 2, 65, 0, 1), (neg, None, 2, 2, 0, 1),
                 (n, None, 2, 2, -1, 1), (n, None, 2, 2, 0, 0), (n, bad_sub, 2, 2, 0, 1),
                 (None, None, 2, 2, 0, 1), (n, None, -1, 2, 0, 1)]:
        assert zero3.raw_status("zero3_partition", *args, C.byref(out)) == zero3.EINVAL, args
    assert zero3.raw_status("zero3_partition", n, None, 2, 2, 0, 1, None) == zero3.EINVAL


FAKE = 1 << 20       # a 16-byte aligned fake device address (never dereferenced)
MISALIGNED = FAKE + 2


def _plan(nd=2):
    from zero_sharded_optimizer_shard_gb300 import zero3
    return zero3.Plan([1000, 10, 2000], [0, 0, 1], nd, threshold=100, bucket=512)


def test_step_rejects_bad_arguments_before_any_launch(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    p = _plan()
    hp = zero3.hparams()
    lo, hi = 0, p.info.psi_pad
    ok = [FAKE, FAKE]
    P = zero3._ptrs

    def step(t=1, grads=ok, origin=0, master=ok, m=ok, v=ok, sparam=ok, full=FAKE, lo=lo, hi=hi,
             hp_=hp):
        return zero3.raw_status("zero3_step", p.handle, C.byref(hp_) if hp_ is not None else None,
                                t, P(grads), origin, P(master), P(m), P(v), P(sparam), full,
                                None, lo, hi, None)

    E = zero3.EINVAL
    assert step(t=0) == E
    assert step(hp_=None) == E
    assert step(hp_=zero3.hparams(beta1=1.0)) == E
    assert step(hp_=zero3.hparams(lr=float("nan"))) == E
    assert step(hi=hi + 1) == E
    assert step(lo=5, hi=4) == E
    assert step(origin=1) == E
    assert step(grads=[FAKE, 0]) == E                  # a missing rank
    assert step(grads=[FAKE, MISALIGNED]) == E
    assert step(grads=None) == E
    assert step(master=[FAKE, 0]) == E
    assert step(v=[MISALIGNED, FAKE]) == E
    assert step(sparam=[FAKE, MISALIGNED]) == E
    assert step(full=0) == E
    assert step(full=MISALIGNED) == E
    # a rank outside the range may pass NULL state, but the range here covers
    # both ranks
    assert step(lo=0, hi=p.info.shard_len, master=[FAKE, 0], full=MISALIGNED) == E
    # the persistent group is validated before the main launch
    ps = zero3.persist_state([FAKE, 0], FAKE, FAKE, FAKE, FAKE)
    st = zero3.raw_status("zero3_step", p.handle, C.byref(hp), 1, P(ok), 0, P(ok), P(ok), P(ok),
                          P(ok), FAKE, C.byref(ps), lo, hi, None)
    assert st == E


def test_unfused_calls_reject_bad_arguments(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    p = _plan(3)
    hp = zero3.hparams()
    ok = [FAKE] * 3
    P = zero3._ptrs
    hi = p.info.psi_pad
    E = zero3.EINVAL
    assert zero3.raw_status("zero3_reduce_scatter", p.handle, P(ok), 0, 0, hi, P(ok), 7,
                            None) == E
    assert zero3.raw_status("zero3_reduce_scatter", p.handle, P([FAKE, FAKE, 0]), 0, 0, hi, P(ok),
                            zero3.F32, None) == E
    assert zero3.raw_status("zero3_adamw_step", p.handle, C.byref(hp), 1, P(ok), zero3.F32,
                            P(ok), P(ok), P(ok), P([FAKE, MISALIGNED, FAKE]), 0, hi, None) == E
    assert zero3.raw_status("zero3_allgather", p.handle, P(ok), MISALIGNED, 0, hi, None) == E
    assert zero3.raw_status("zero3_cast_params", p.handle, P(ok), P(ok), MISALIGNED, None, 0, hi,
                            None) == E
    # empty ranges are no-ops and need no pointers
    assert zero3.raw_status("zero3_allgather", p.handle, None, 0, 3, 3, None) == zero3.OK
    assert zero3.raw_status("zero3_reduce_scatter", p.handle, None, 0, 0, 0, None, zero3.F32,
                            None) == zero3.OK


def test_submodule_state_errors_on_host(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    p = _plan()
    assert zero3.zero3_submodule_status(p, 0) == zero3.NOT_AVAILABLE
    with pytest.raises(zero3.Zero3Error) as e:
        zero3.zero3_release_submodule(p, 0)
    assert e.value.status == zero3.ESTATE
    with pytest.raises(zero3.Zero3Error) as e:
        zero3.zero3_submodule_wait(p, 1)
    assert e.value.status == zero3.ESTATE
    for bad in (-1, 2):
        with pytest.raises(zero3.Zero3Error) as e:
            zero3.zero3_submodule_status(p, bad)
        assert e.value.status == zero3.EINVAL
    # misaligned output or a missing owner shard is rejected before any work
    st = zero3.raw_status("zero3_fetch_submodule", p.handle, 0, zero3._ptrs([FAKE, FAKE]), FAKE,
                          MISALIGNED, None)
    assert st == zero3.EINVAL
    st = zero3.raw_status("zero3_fetch_submodule", p.handle, 1, zero3._ptrs([FAKE, 0]), FAKE,
                          FAKE, None)
    assert st == zero3.EINVAL
    assert zero3.zero3_submodule_status(p, 0) == zero3.NOT_AVAILABLE


def test_fetch_submodules_rejects_bad_arguments_on_host(lib):
    """The multi-submodule fetch checks every listed submodule before it
    launches anything or changes any state (fake device pointers: a launch
    would fault, so none may happen)."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    p = _plan()
    P = zero3._ptrs
    ks = (C.c_int32 * 3)(0, 1, 2)
    E = zero3.EINVAL
    f = lambda k, n, sp, outs: zero3.raw_status("zero3_fetch_submodules", p.handle, k, n, sp, FAKE,
                                                outs, None)
    assert f(ks, 2, P([FAKE, FAKE]), P([FAKE, MISALIGNED])) == E     # second output misaligned
    assert f(ks, 3, P([FAKE, FAKE]), P([FAKE, FAKE, FAKE])) == E     # id 2 out of range
    assert f(ks, -1, P([FAKE, FAKE]), P([FAKE])) == E
    assert f(ks, 2, P([FAKE, FAKE]), None) == E
    assert f(None, 2, P([FAKE, FAKE]), P([FAKE, FAKE])) == E
    assert f(ks, 2, P([FAKE, 0]), P([FAKE, FAKE])) == E              # a missing owner shard
    assert f(None, 0, None, None) == zero3.OK                         # nothing to do
    for k in (0, 1):
        assert zero3.zero3_submodule_status(p, k) == zero3.NOT_AVAILABLE


def test_status_strings(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    assert zero3.status_string(zero3.OK) == "ok"
    assert "invalid" in zero3.status_string(zero3.EINVAL)
    assert zero3.status_string(99) == "unknown status"


# ---------------------------------------------------------------- checkpoint headers
def _header(kind=1, rank=0, n_ranks=2, n_elems=None, t=5, fp=None, magic=b"ZERO3CKP", version=1,
            plan=None):
    import struct
    return struct.pack("<8sIIiiqqQ", magic, version, kind, rank, n_ranks,
                       n_elems if n_elems is not None else plan.info.shard_len, t,
                       fp if fp is not None else 0)


def test_checkpoint_load_rejects_bad_files(lib, tmp_path):
    """Every header mismatch is reported as ZERO3_EIO before any device memory
    is touched (the device pointers here are fake)."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    p = _plan()
    t = C.c_int64()
    cases = {
        "missing": None,
        "short": b"ZERO3C",
        "magic": _header(magic=b"NOTZERO3", plan=p),
        "fingerprint": _header(fp=12345, plan=p),
        "version": _header(version=2, plan=p),
        "kind": _header(kind=3, plan=p),
        "rank": _header(rank=1, plan=p),
        "n_elems": _header(n_elems=7, plan=p),
    }
    for name, data in cases.items():
        path = tmp_path / f"{name}.ckpt"
        if data is not None:
            path.write_bytes(data)
        st = zero3.raw_status("zero3_load_shard", p.handle, 0, C.byref(t), FAKE, FAKE, FAKE,
                              str(path).encode(), None)
        assert st == zero3.EIO, name
    # argument errors come first
    assert zero3.raw_status("zero3_load_shard", p.handle, 2, C.byref(t), FAKE, FAKE, FAKE,
                            b"x", None) == zero3.EINVAL
    assert zero3.raw_status("zero3_save_shard", p.handle, 0, -1, FAKE, FAKE, FAKE, b"x",
                            None) == zero3.EINVAL
    assert zero3.raw_status("zero3_save_16bit_weights", p.handle, MISALIGNED, FAKE, b"x",
                            None) == zero3.EINVAL


def test_coordinator_create_rejects_bad_arguments(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    p = _plan()
    out = C.c_void_p()
    big = p.submodule(1)[1]
    cfg = zero3.PrefetchConfig(10**6, 10**6, 10**6)
    P = zero3._ptrs
    S1, S2 = 0x1000, 0x2000  # two distinct stream handles (never used: creation fails first)

    def create(trace=(0, 1), sparam=(FAKE, FAKE), persist=FAKE, arena=FAKE, n=big, cfg_=cfg,
               s1=S1, s2=S2):
        tr = (C.c_int32 * max(len(trace), 1))(*trace)
        return zero3.raw_status("zero3_coordinator_create", p.handle, tr, len(trace),
                                P(list(sparam)) if sparam is not None else None, persist, arena,
                                n, C.byref(cfg_) if cfg_ is not None else None, s1, s2,
                                C.byref(out))
    E = zero3.EINVAL
    assert create(n=big - 1) == E                       # arena below the largest submodule
    assert create(cfg_=zero3.PrefetchConfig(0, big - 1, 0)) == E  # live budget too small
    assert create(cfg_=zero3.PrefetchConfig(-1, big, 0)) == E
    assert create(cfg_=None) == E
    assert create(s2=S1) == E                           # same stream twice
    assert create(trace=(0, 2)) == E                    # unknown submodule
    assert create(sparam=(FAKE, 0)) == E                # missing shard
    assert create(sparam=None) == E
    assert create(arena=MISALIGNED) == E
    assert create(persist=0) == E                       # submodule 0 holds a persistent tensor


# ---------------------------------------------------------------- offline merge and plan memory
def _fnv1a(values):
    h = 14695981039346656037
    for x in values:
        for b in int(x).to_bytes(8, "little", signed=True):
            h ^= b
            h = (h * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return h


def _write(path, kind, rank, nd, n, t, fp, arrays):
    import struct
    with open(path, "wb") as f:
        f.write(struct.pack("<8sIIiiqqQ", b"ZERO3CKP", 1, kind, rank, nd, n, t, fp))
        for a in arrays:
            f.write(np.ascontiguousarray(a, np.float32).tobytes())


def test_merge_shards_matches_oracle(lib, tmp_path):
    """Shard files written from the documented format (host only) are
    merged by the library into the oracle's consolidated fp32 weights."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.ragged_small(7)
    ref = O.partition(w.numels, w.submodule_of, 7, w.threshold, w.bucket)
    p = zero3.Plan(w.numels, w.submodule_of, 7, w.threshold, w.bucket)
    fp = _fnv1a([7, w.threshold, len(w.numels)] + list(w.numels))
    rng = np.random.default_rng(0)
    masters = [rng.standard_normal(ref.shard_len).astype(np.float32) for _ in range(7)]
    pm = rng.standard_normal(ref.psi_s).astype(np.float32)
    paths = []
    for r in range(7):
        paths.append(tmp_path / f"r{r}.ckpt")
        _write(paths[-1], 1, r, 7, ref.shard_len, 9, fp,
               [masters[r], np.zeros(ref.shard_len), np.ones(ref.shard_len)])
    _write(tmp_path / "p.ckpt", 2, -1, 7, ref.psi_s, 9, fp, [pm, np.zeros(ref.psi_s), np.zeros(ref.psi_s)])
    out = tmp_path / "merged.bin"
    zero3.zero3_merge_shards(p, paths, tmp_path / "p.ckpt", out)
    raw = out.read_bytes()
    import struct
    magic, ver, kind, rank, nd, n, t, fph = struct.unpack_from("<8sIIiiqqQ", raw)
    assert (magic, ver, kind, nd, n, t, fph) == (b"ZERO3CKP", 1, 4, 7, sum(w.numels), 9, fp)
    got = np.frombuffer(raw, np.float32, offset=48)
    want = np.concatenate(O.merge_fp32_weights(ref, masters, pm))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # a shard of another step, a missing rank file, or a wrong rank: EIO, no output
    _write(paths[3], 1, 3, 7, ref.shard_len, 8, fp, [masters[3]] * 3)
    out2 = tmp_path / "merged2.bin"
    with pytest.raises(zero3.Zero3Error) as exc:
        zero3.zero3_merge_shards(p, paths, tmp_path / "p.ckpt", out2)
    assert exc.value.status == zero3.EIO and not out2.exists()
    swapped = list(paths)
    swapped[1], swapped[2] = swapped[2], swapped[1]
    with pytest.raises(zero3.Zero3Error):
        zero3.zero3_merge_shards(p, swapped, tmp_path / "p.ckpt", out2)
    with pytest.raises(zero3.Zero3Error):
        zero3.zero3_merge_shards(p, paths[:6] + [tmp_path / "nope"], tmp_path / "p.ckpt", out2)
    # a shard file one element short, or with one byte too many: EIO, no output
    _write(paths[3], 1, 3, 7, ref.shard_len, 9, fp, [masters[3], np.zeros(ref.shard_len),
                                                     np.ones(ref.shard_len)])
    full3 = paths[3].read_bytes()
    for bad in (full3[:-4], full3 + b"\0"):
        paths[3].write_bytes(bad)
        with pytest.raises(zero3.Zero3Error) as exc:
            zero3.zero3_merge_shards(p, paths, tmp_path / "p.ckpt", out2)
        assert exc.value.status == zero3.EIO and not out2.exists()


_ATOMIC_CHILD = r'''
import os, resource, signal, sys
sys.path.insert(0, {root!r})
import numpy as np
from zero_sharded_optimizer_shard_gb300 import workloads as W, zero3
from tests.test_abi_host import _fnv1a, _write
w = W.ragged_small(7)
p = zero3.Plan(w.numels, w.submodule_of, 7, w.threshold, w.bucket)
info = p.info
fp = _fnv1a([7, w.threshold, len(w.numels)] + list(w.numels))
d = {d!r}
paths = [os.path.join(d, "r%d.ckpt" % r) for r in range(7)]
for r in range(7):
    _write(paths[r], 1, r, 7, info.shard_len, 1, fp, [np.full(info.shard_len, r, np.float32)] * 3)
_write(os.path.join(d, "p.ckpt"), 2, -1, 7, info.psi_s, 1, fp, [np.zeros(info.psi_s)] * 3)
out = os.path.join(d, "merged.bin")
# files larger than 64 KiB cannot be written from here on: the merge fails
# in the middle of writing its output
signal.signal(signal.SIGXFSZ, signal.SIG_IGN)
resource.setrlimit(resource.RLIMIT_FSIZE, (1 << 16, 1 << 16))
try:
    zero3.zero3_merge_shards(p, paths, os.path.join(d, "p.ckpt"), out)
except zero3.Zero3Error as e:
    print("status", e.status)
'''


def test_failed_save_keeps_the_previous_file(lib, tmp_path):
    """A save that fails in the middle of writing (here: the process may
    not write files beyond 64 KiB) reports EIO, leaves the file that was at
    the destination path byte for byte, and leaves no temporary file."""
    import subprocess
    import sys
    from zero_sharded_optimizer_shard_gb300 import zero3
    out = tmp_path / "merged.bin"
    out.write_bytes(b"previous checkpoint")
    code = _ATOMIC_CHILD.format(root=ROOT, d=str(tmp_path))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert f"status {zero3.EIO}" in r.stdout, r.stdout + r.stderr
    assert out.read_bytes() == b"previous checkpoint"
    assert sorted(x.name for x in tmp_path.iterdir() if ".tmp." in x.name) == []


def test_plan_memory_bytes_matches_oracle(lib):
    from zero_sharded_optimizer_shard_gb300 import zero3
    for name in ("toy_mlp", "gpt2_small", "decoder_1p3b", "llama_7b_rank0", "ragged"):
        w = W.BY_NAME[name]()
        ref = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
        p = zero3.Plan(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
        for stage in range(4):
            assert zero3.zero3_plan_memory_bytes(p, stage) == pytest.approx(
                O.plan_memory_bytes(ref, stage), rel=1e-15)
