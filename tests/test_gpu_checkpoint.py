"""Checkpoint save/resume of the shards and the consolidated 16-bit weights,
through the C ABI, against the oracle."""
import struct

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from tests._oracle_runs import bits, f32, oracle_run, u16  # noqa: E402
from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu

HEADER = struct.Struct("<8sIIiiqqQ")


def make(w):
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    e = Emulation(w)
    e.init_params()
    return e


def steps(e, t0, t1):
    for t in range(t0, t1 + 1):
        e.fill_grads(t)
        e.step(t)


def save_all(e, t, d):
    from zero_sharded_optimizer_shard_gb300 import zero3
    for r in range(e.nd):
        zero3.zero3_save_shard(e.plan, r, t, e.master[r].data_ptr(), e.m[r].data_ptr(),
                               e.v[r].data_ptr(), d / f"rank{r}.ckpt", e.sid)
    zero3.zero3_save_persistent(e.plan, t, e.persist, d / "persistent.ckpt", e.sid)


def load_all(e, d):
    from zero_sharded_optimizer_shard_gb300 import zero3
    ts = {zero3.zero3_load_shard(e.plan, r, e.master[r].data_ptr(), e.m[r].data_ptr(),
                                 e.v[r].data_ptr(), d / f"rank{r}.ckpt", e.sid)
          for r in range(e.nd)}
    ts.add(zero3.zero3_load_persistent(e.plan, e.persist, d / "persistent.ckpt", e.sid))
    assert len(ts) == 1
    # bf16 shards, full buffer and persistent params are bf16(master)
    zero3.zero3_cast_params(e.plan, e.ptrs(e.master), e.ptrs(e.sparam), e.full.data_ptr(),
                            e.persist, 0, e.psi_pad, e.sid)
    return ts.pop()


@pytest.mark.parametrize("wname", ["mini4", "ragged7"])
def test_resume_equals_uninterrupted(tmp_path, wname):
    """5 steps, save, restore into fresh buffers, 5 more steps == 10 steps,
    bit for bit, and both equal the oracle's 10 steps."""
    w = {"mini4": lambda: W.mini_gpt(4), "ragged7": lambda: W.ragged_small(7)}[wname]()
    a = make(w)
    steps(a, 1, 10)
    b = make(w)
    steps(b, 1, 5)
    save_all(b, 5, tmp_path)
    c = make(w)
    for x in c.master + c.m + c.v:
        x.fill_(float("nan"))  # anything the load does not overwrite shows up
    t = load_all(c, tmp_path)
    assert t == 5
    steps(c, 6, 10)
    torch.cuda.synchronize()
    plan, st, full, ps = oracle_run(w, 10)
    for r in range(w.n_ranks):
        for name in ("master", "m", "v"):
            got = f32(getattr(c, name)[r])
            assert np.array_equal(bits(got), bits(f32(getattr(a, name)[r]))), (name, r)
            assert np.array_equal(bits(got), bits(getattr(st, name)[r])), (name, r)
        assert np.array_equal(u16(c.sparam[r]), st.sparam[r])
    assert np.array_equal(u16(c.full), full)
    assert np.array_equal(bits(f32(c.pmaster)), bits(ps.master))
    assert np.array_equal(u16(c.pparam), ps.param)


def test_16bit_weights_file_matches_oracle(tmp_path):
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.ragged_small(7)
    e = make(w)
    steps(e, 1, 3)
    path = tmp_path / "weights16.bin"
    zero3.zero3_save_16bit_weights(e.plan, e.full.data_ptr(), e.pparam.data_ptr(), path, e.sid)
    raw = path.read_bytes()
    magic, ver, kind, rank, nd, n, t, fp = HEADER.unpack_from(raw)
    assert (magic, ver, kind, nd) == (b"ZERO3CKP", 1, 3, 7)
    data = np.frombuffer(raw, np.uint16, offset=HEADER.size)
    assert n == data.size == sum(w.numels)
    plan, st, full, ps = oracle_run(w, 3)
    want = np.concatenate(O.gather_16bit_weights(plan, st.sparam, ps.param))
    assert np.array_equal(data, want)


def test_load_rejects_every_header_mismatch(tmp_path):
    """A real shard file with one header field changed at a time, a
    truncated file and one with trailing bytes: all ZERO3_EIO, and the
    destination buffers stay untouched in every case."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.toy_mlp()
    e = make(w)
    steps(e, 1, 1)
    good = tmp_path / "good.ckpt"
    zero3.zero3_save_shard(e.plan, 0, 1, e.master[0].data_ptr(), e.m[0].data_ptr(),
                           e.v[0].data_ptr(), good, e.sid)
    raw = bytearray(good.read_bytes())
    assert len(raw) == HEADER.size + 3 * 4 * e.S
    fields = HEADER.unpack_from(raw)
    dst = [torch.full((e.S,), 7.0, device="cuda") for _ in range(3)]
    variants = {}
    for k, name in enumerate(["magic", "version", "kind", "rank", "n_ranks", "n_elems", "t", "fp"]):
        f = list(fields)
        f[k] = b"ZERO3CKQ" if k == 0 else (-1 if k == 6 else f[k] + 1)
        variants[name] = HEADER.pack(*f) + raw[HEADER.size:]
    variants["truncated"] = bytes(raw[:-4])
    variants["trailing"] = bytes(raw) + b"\0"
    for name, data in variants.items():
        p = tmp_path / f"{name}.ckpt"
        p.write_bytes(data)
        with pytest.raises(zero3.Zero3Error) as exc:
            zero3.zero3_load_shard(e.plan, 0, *[d.data_ptr() for d in dst], p, e.sid)
        assert exc.value.status == zero3.EIO, name
        # rejected before any byte reaches the device, whatever was wrong
        assert all(bool((d == 7.0).all()) for d in dst), name
    # the unmodified file loads, into the right rank only
    t = zero3.zero3_load_shard(e.plan, 0, *[d.data_ptr() for d in dst], good, e.sid)
    assert t == 1 and torch.equal(dst[0], e.master[0])
    with pytest.raises(zero3.Zero3Error):
        zero3.zero3_load_shard(e.plan, 1, *[d.data_ptr() for d in dst], good, e.sid)
    other = zero3.Plan(w.numels, w.submodule_of, 4, w.threshold, w.bucket)
    with pytest.raises(zero3.Zero3Error):
        zero3.zero3_load_shard(other, 0, *[d.data_ptr() for d in dst], good, e.sid)


def test_merge_saved_shards_matches_oracle(tmp_path):
    """Shards saved by the library after 3 steps, merged offline into
    complete fp32 tensors == the oracle's masters merged the same way."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.ragged_small(7)
    e = make(w)
    steps(e, 1, 3)
    save_all(e, 3, tmp_path)
    out = tmp_path / "merged.bin"
    zero3.zero3_merge_shards(e.plan, [tmp_path / f"rank{r}.ckpt" for r in range(7)],
                             tmp_path / "persistent.ckpt", out)
    raw = out.read_bytes()
    magic, ver, kind, rank, nd, n, t, fp = HEADER.unpack_from(raw)
    assert (kind, n, t) == (4, sum(w.numels), 3)
    got = np.frombuffer(raw, np.float32, offset=HEADER.size)
    plan, st, full, ps = oracle_run(w, 3)
    want = np.concatenate(O.merge_fp32_weights(plan, st.master, ps.master))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
