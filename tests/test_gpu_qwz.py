"""qwZ (quantized parameter all-gather) through the C ABI against the oracle:
the fused step's states and shards, its int8 codes and block scales, and
the dequantizing all-gather, bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from tests._oracle_runs import bits as b32, f32, host_grads, host_master, u16  # noqa: E402
from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


def wire(e):
    nb = -(-e.S // 256)
    codes = [torch.zeros(max(e.S, 16), dtype=torch.int8, device="cuda") for _ in range(e.nd)]
    scales = [torch.zeros(max(nb, 4), dtype=torch.float32, device="cuda") for _ in range(e.nd)]
    return codes, scales


def i8(t):
    return t.detach().cpu().numpy().view(np.int8)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("wname", ["mini2", "mini3", "mini8", "ragged7"])
def test_qwz_step_and_allgather_match_oracle(wname, bits):
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    w = {"mini2": lambda: W.mini_gpt(2), "mini3": lambda: W.mini_gpt(3),
         "mini8": lambda: W.mini_gpt(8), "ragged7": lambda: W.ragged_small(7)}[wname]()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e = Emulation(w)
    e.init_params()
    codes, scales = wire(e)
    mf, mp = host_master(w, plan)
    st, full, _ = O.init_state(plan, mf, mp)
    for t in range(1, 4):
        e.fill_grads(t)
        zero3.zero3_step_qwz(e.plan, e.hp, t, e.ptrs(e.grads[0]), 0, e.ptrs(e.master), e.ptrs(e.m),
                             e.ptrs(e.v), e.ptrs(e.sparam), e.ptrs(codes), e.ptrs(scales), None,
                             0, e.psi_pad, e.sid, bits=bits)
        zero3.zero3_allgather_qwz(e.plan, e.ptrs(codes), e.ptrs(scales), e.full.data_ptr(), 0,
                                  e.psi_pad, e.sid, bits=bits)
        O.sharded_step(plan, w.hparams, t, host_grads(w, plan, t), st, full)
    torch.cuda.synchronize()
    q = [O.qwz_quantize(st.sparam[r], bits=bits) for r in range(w.n_ranks)]
    nbytes = -(-e.S * bits // 8)
    for r in range(w.n_ranks):
        assert np.array_equal(b32(f32(e.master[r])), b32(st.master[r]))
        assert np.array_equal(u16(e.sparam[r]), st.sparam[r])
        wire_bytes = i8(codes[r])[:nbytes].view(np.uint8)
        assert np.array_equal(wire_bytes, O.qwz_pack(q[r][0], bits)), f"codes rank {r}"
        assert np.array_equal(b32(f32(scales[r])[:q[r][1].size]), b32(q[r][1])), f"scales {r}"
    want = O.qwz_allgather(plan, [c for c, _ in q], [s for _, s in q])
    assert np.array_equal(u16(e.full), want)


def test_quantize_shards_and_partial_ranges():
    """Standalone quantization == oracle; a block-aligned sub-range touches
    only its blocks; a range that cuts a block is rejected; the dequantizing
    gather accepts any range."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    w = W.mini_gpt(3)
    e = Emulation(w)
    e.init_params()
    codes, scales = wire(e)
    S = e.S
    zero3.zero3_quantize_shards(e.plan, e.ptrs(e.sparam), e.ptrs(codes), e.ptrs(scales), 0,
                                e.psi_pad, e.sid)
    torch.cuda.synchronize()
    for r in range(3):
        c, s = O.qwz_quantize(u16(e.sparam[r]))
        assert np.array_equal(i8(codes[r])[:S], c)
        assert np.array_equal(b32(f32(scales[r])[:s.size]), b32(s))
    # sub-range: rank 1's blocks 2..5 only
    for x in codes:
        x.zero_()
    zero3.zero3_quantize_shards(e.plan, e.ptrs(e.sparam), e.ptrs(codes), e.ptrs(scales),
                                S + 512, S + 1536, e.sid)
    torch.cuda.synchronize()
    c1, _ = O.qwz_quantize(u16(e.sparam[1]))
    got = i8(codes[1])
    assert np.array_equal(got[512:1536], c1[512:1536])
    assert not got[:512].any() and not got[1536:S].any() and not i8(codes[0]).any()
    for bad in [(S + 100, S + 1536), (S + 512, S + 1000)]:
        with pytest.raises(zero3.Zero3Error) as exc:
            zero3.zero3_quantize_shards(e.plan, e.ptrs(e.sparam), e.ptrs(codes), e.ptrs(scales),
                                        *bad, e.sid)
        assert exc.value.status == zero3.EINVAL
    # dequantize an odd range only (codes of every shard quantized again first)
    zero3.zero3_quantize_shards(e.plan, e.ptrs(e.sparam), e.ptrs(codes), e.ptrs(scales), 0,
                                e.psi_pad, e.sid)
    e.full.zero_()
    lo, hi = S - 13, 2 * S + 7
    zero3.zero3_allgather_qwz(e.plan, e.ptrs(codes), e.ptrs(scales), e.full.data_ptr(), lo, hi,
                              e.sid)
    torch.cuda.synchronize()
    got = u16(e.full)
    assert not got[:lo].any() and not got[hi:].any()
    c0, s0 = O.qwz_quantize(u16(e.sparam[0]))
    c1, s1 = O.qwz_quantize(u16(e.sparam[1]))
    c2, s2 = O.qwz_quantize(u16(e.sparam[2]))
    assert np.array_equal(got[lo:S], O.qwz_dequantize(c0, s0)[lo:S])
    assert np.array_equal(got[S:2 * S], O.qwz_dequantize(c1, s1))
    assert np.array_equal(got[2 * S:hi], O.qwz_dequantize(c2, s2)[:hi - 2 * S])


def test_qwz_rejects_other_widths():
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    e = Emulation(W.toy_mlp())
    e.init_params()
    codes, scales = wire(e)
    for b in (0, 2, 16):
        with pytest.raises(zero3.Zero3Error) as exc:
            zero3.zero3_quantize_shards(e.plan, e.ptrs(e.sparam), e.ptrs(codes), e.ptrs(scales), 0,
                                        e.psi_pad, e.sid, bits=b)
        assert exc.value.status == zero3.EINVAL


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("wname", ["ragged7", "mini8"])
def test_dequantizing_gather_of_sub_ranges(wname, bits):
    """The dequantizing all-gather over many sub-ranges of the flat buffer:
    the whole range, single elements, ranges around every rank boundary,
    ranges ending 1..2053 elements after a shard's start or before its end
    (the last source units of a piece), and seeded random ranges.  On the
    ragged list at N_d = 7 (S mod 8 = 5) every launch has phased sources;
    at N_d = 8 they are aligned.  Each range equals the oracle's whole gather
    there, bit for bit, and no element outside it is written."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    w = {"ragged7": lambda: W.ragged_small(7), "mini8": lambda: W.mini_gpt(8)}[wname]()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e = Emulation(w)
    e.init_params()
    codes, scales = wire(e)
    zero3.zero3_quantize_shards(e.plan, e.ptrs(e.sparam), e.ptrs(codes), e.ptrs(scales), 0,
                                e.psi_pad, e.sid, bits=bits)
    torch.cuda.synchronize()
    q = [O.qwz_quantize(u16(e.sparam[r]), bits=bits) for r in range(e.nd)]
    want = O.qwz_allgather(plan, [c for c, _ in q], [s for _, s in q])
    S, N = e.S, e.psi_pad
    ranges = [(0, N), (0, 1), (N - 1, N)]
    for r in range(e.nd):
        b0, b1 = r * S, (r + 1) * S
        ranges += [(b0 - 9, b0 + 9), (b0 - 1, b0 + 1), (b0 - 3, b0), (b0, b0 + 5)]
        ranges += [(b0, b0 + d) for d in (1, 7, 8, 9, 2053)]
        ranges += [(b1 - d, b1) for d in (1, 7, 8, 9, 2053)]
    rng = np.random.default_rng(7)
    for _ in range(24):
        lo = int(rng.integers(0, N))
        ranges.append((lo, lo + int(rng.integers(1, 5000))))
    ranges = sorted({(max(0, lo), min(N, hi)) for lo, hi in ranges if min(N, hi) > max(0, lo)})
    for lo, hi in ranges:
        e.full.view(torch.int16).fill_(0x7FC1)
        zero3.zero3_allgather_qwz(e.plan, e.ptrs(codes), e.ptrs(scales), e.full.data_ptr(), lo,
                                  hi, e.sid, bits=bits)
        torch.cuda.synchronize()
        got = u16(e.full)
        assert np.array_equal(got[lo:hi], want[lo:hi]), (lo, hi)
        assert (got[:lo] == 0x7FC1).all() and (got[hi:] == 0x7FC1).all(), (lo, hi)
