"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, element by element, at sizes the oracle finishes in
seconds.  Floating point: the library is built to reproduce the oracle's
operation order, so results are compared bit for bit, and additionally
against the stated tolerance (2e-6 relative on fp32 master/m/v, 1 bf16 ulp
on parameters)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from tests._oracle_runs import (assert_bf16_close, assert_f32_close, bits, f32,  # noqa: E402
                                host_grads, oracle_run, sampled_oracle, u16)
from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda:0")


def make_emu(w, **kw):
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    e = Emulation(w, **kw)
    e.init_params()
    return e


def run_device(w, T, grad_step=None, **kw):
    e = make_emu(w, **kw)
    for t in range(1, T + 1):
        e.fill_grads(t if grad_step is None else grad_step)
        e.step(t)
    torch.cuda.synchronize()
    return e


def compare_all(e, plan, st, full, ps, bitwise=True):
    for r in e.state_ranks:
        for name, got, ref in (("master", e.master[r], st.master[r]), ("m", e.m[r], st.m[r]),
                               ("v", e.v[r], st.v[r])):
            g = f32(got)
            assert_f32_close(g, ref, what=f"{name}[{r}]")
            if bitwise:
                assert np.array_equal(bits(g), bits(ref)), f"{name}[{r}] not bit-exact"
        assert_bf16_close(u16(e.sparam[r]), st.sparam[r], what=f"sparam[{r}]")
        if bitwise:
            assert np.array_equal(u16(e.sparam[r]), st.sparam[r]), f"sparam[{r}]"
    lo = min(e.state_ranks) * e.S
    hi = (max(e.state_ranks) + 1) * e.S
    assert np.array_equal(u16(e.full)[lo:hi], full[lo:hi]), "full"
    for name, got, ref in (("pmaster", e.pmaster, ps.master), ("pm", e.pm, ps.m),
                           ("pv", e.pv, ps.v)):
        g = f32(got)
        assert_f32_close(g, ref, what=name)
        if bitwise:
            assert np.array_equal(bits(g), bits(ref)), name
    assert np.array_equal(u16(e.pparam), ps.param), "pparam"


# ---------------------------------------------------------------- generator
def test_device_generator_matches_host(dev):
    from zero_sharded_optimizer_shard_gb300 import synth, synth_device
    n, i0 = 1 << 20, 123_456_789
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    synth_device.normal(out.data_ptr(), n, seed=9, stream_id=3, step=4, rank=5, index0=i0,
                        sigma=1e-3, outlier_p=0.01, outlier_sigma=0.1)
    ref = synth.normal_bf16(9, 3, 4, 5, np.arange(i0, i0 + n), 1e-3, 0.01, 0.1)
    assert np.array_equal(u16(out), ref)
    outf = torch.empty(n, dtype=torch.float32, device=dev)
    synth_device.normal(outf.data_ptr(), n, seed=2, stream_id=1, step=0, rank=0, index0=0,
                        sigma=0.02, bf16=False)
    assert np.array_equal(bits(f32(outf)), bits(synth.normal_f32(2, 1, 0, 0, np.arange(n), 0.02)))


# ---------------------------------------------------------------- fused step
@pytest.mark.parametrize("wname,T", [("toy", 3), ("mini4", 10), ("ragged7", 5)])
def test_fused_step_matches_oracle(dev, wname, T):
    w = {"toy": W.toy_mlp, "mini4": lambda: W.mini_gpt(4), "ragged7": lambda: W.ragged_small(7)}[wname]()
    plan, st, full, ps = oracle_run(w, T)
    e = run_device(w, T)
    compare_all(e, plan, st, full, ps)


@pytest.mark.parametrize("nd", [1, 2, 3, 5, 6, 8, 9, 16, 33, 64])
def test_fused_step_rank_counts(dev, nd):
    """Specialised (1, 2, 4, 8) and generic rank counts; S not a multiple of 8
    for most of them, so both the vector and the element paths run; 33 and 64
    run the generic path with a partial last group of ranks and the maximum."""
    if nd <= 16:
        w = W.mini_gpt(nd)
    else:
        w = W.Workload(f"small_nd{nd}", [150_001, 123_457, 99_999, 7, 180_000], [0, 0, 1, 1, 2],
                       n_ranks=nd, steps=3, seed=13)
    w.steps = 3
    plan, st, full, ps = oracle_run(w, 3)
    e = run_device(w, 3)
    compare_all(e, plan, st, full, ps)


def test_bucketed_launches_equal_one_launch(dev):
    """Per-bucket launches with bucket-sized gradient buffers (grads_origin =
    bucket start) give the same bits as one launch over the whole range."""
    w = W.mini_gpt(3)
    w.bucket = 100_003  # odd bucket edges inside shards
    plan, st, full, ps = oracle_run(w, 3)
    e = run_device(w, 3, bucketed=True)
    assert len(e.chunks) > 3
    compare_all(e, plan, st, full, ps)


def test_rank0_view_matches_oracle(dev):
    """Only rank 0 holds optimizer state (NULL state pointers for the other
    ranks); bucketed gradient buffers cover rank 0's range only."""
    w = W.mini_gpt(4)
    w.bucket = 150_000
    plan, st, full, ps = oracle_run(w, 4)
    e = run_device(w, 4, state_ranks=[0], bucketed=True)
    compare_all(e, plan, st, full, ps)


def test_padding_stays_exactly_zero(dev):
    w = W.ragged_small(7)
    plan = O.partition(w.numels, w.submodule_of, 7, w.threshold, w.bucket)
    assert plan.psi_pad > plan.psi_p
    e = run_device(w, 3)
    S = e.S
    r = plan.psi_p // S
    tail = f32(e.master[r])[plan.psi_p - r * S:]
    assert tail.size and not bits(tail).any()
    assert not u16(e.full)[plan.psi_p:].any()
    assert not bits(f32(e.m[r])[plan.psi_p - r * S:]).any()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_subranges(dev, seed):
    """Random sub-ranges [lo, hi): ranges inside one shard, across shard
    boundaries, single elements and empty ranges, compared with the oracle on
    the same range; elements outside the range must stay untouched."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    rng = np.random.default_rng(seed)
    w = W.mini_gpt(5)
    plan = O.partition(w.numels, w.submodule_of, 5, w.threshold, w.bucket)
    e = make_emu(w)
    e.fill_grads(1)
    from tests._oracle_runs import host_master
    mf, mp = host_master(w, plan)
    st, full, _ = O.init_state(plan, mf, mp)
    G = host_grads(w, plan, 1)
    ranges = [(0, 0), (17, 18), (plan.shard_len - 3, plan.shard_len + 5), (plan.psi_pad - 1, plan.psi_pad)]
    for _ in range(6):
        a, b = sorted(int(x) for x in rng.integers(0, plan.psi_pad + 1, 2))
        ranges.append((a, b))
    for t, (a, b) in enumerate(ranges, start=1):
        zero3.zero3_step(e.plan, e.hp, t, e.ptrs(e.grads[0]), 0, e.ptrs(e.master), e.ptrs(e.m),
                         e.ptrs(e.v), e.ptrs(e.sparam), e.full.data_ptr(), None, a, b, e.sid)
        O.sharded_step(plan, w.hparams, t, G, st, full, a, b)
    torch.cuda.synchronize()
    for r in range(5):
        assert np.array_equal(bits(f32(e.master[r])), bits(st.master[r]))
        assert np.array_equal(bits(f32(e.v[r])), bits(st.v[r]))
        assert np.array_equal(u16(e.sparam[r]), st.sparam[r])
    assert np.array_equal(u16(e.full), full)


# ---------------------------------------------------------------- unfused calls
@pytest.mark.parametrize("nd", [2, 4, 7])
def test_unfused_f32_equals_fused(dev, nd):
    """reduce_scatter(F32) + adamw_step(F32) + allgather == fused step, bit for bit."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.mini_gpt(nd)
    a = make_emu(w)
    b = make_emu(w)
    shard_g = [torch.empty(a.S, dtype=torch.float32, device=dev) for _ in range(nd)]
    for t in range(1, 4):
        a.fill_grads(t)
        b.fill_grads(t)
        a.step(t, with_persistent=False)
        lo, hi = b.chunks[0]
        zero3.zero3_reduce_scatter(b.plan, b.ptrs(b.grads[0]), lo, lo, hi, b.ptrs(shard_g),
                                   zero3.F32, b.sid)
        zero3.zero3_adamw_step(b.plan, b.hp, t, b.ptrs(shard_g), zero3.F32, b.ptrs(b.master),
                               b.ptrs(b.m), b.ptrs(b.v), b.ptrs(b.sparam), lo, hi, b.sid)
        zero3.zero3_allgather(b.plan, b.ptrs(b.sparam), b.full.data_ptr(), lo, hi, b.sid)
    torch.cuda.synchronize()
    for r in range(nd):
        assert np.array_equal(bits(f32(a.master[r])), bits(f32(b.master[r])))
        assert np.array_equal(bits(f32(a.m[r])), bits(f32(b.m[r])))
        assert np.array_equal(bits(f32(a.v[r])), bits(f32(b.v[r])))
        assert np.array_equal(u16(a.sparam[r]), u16(b.sparam[r]))
    assert np.array_equal(u16(a.full), u16(b.full))


def test_reduce_scatter_bf16_and_adam_bf16_match_oracle(dev):
    """Reduce-scatter to a 2-byte shard gradient (rounded to nearest even)
    then AdamW from it, against the oracle's same stages."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    nd = 3
    w = W.mini_gpt(nd)
    plan = O.partition(w.numels, w.submodule_of, nd, w.threshold, w.bucket)
    e = make_emu(w)
    from tests._oracle_runs import host_master
    mf, mp = host_master(w, plan)
    st, full, _ = O.init_state(plan, mf, mp)
    shard_g = [torch.empty(e.S, dtype=torch.bfloat16, device=dev) for _ in range(nd)]
    lo, hi = e.chunks[0]
    for t in range(1, 4):
        e.fill_grads(t)
        zero3.zero3_reduce_scatter(e.plan, e.ptrs(e.grads[0]), lo, lo, hi, e.ptrs(shard_g),
                                   zero3.BF16, e.sid)
        zero3.zero3_adamw_step(e.plan, e.hp, t, e.ptrs(shard_g), zero3.BF16, e.ptrs(e.master),
                               e.ptrs(e.m), e.ptrs(e.v), e.ptrs(e.sparam), lo, hi, e.sid)
        sc = O.adamw_scalars(w.hparams, t, nd)
        gs = O.reduce_scatter(plan, host_grads(w, plan, t), sc["inv_nd"])
        torch.cuda.synchronize()
        for r in range(nd):
            g16 = O.bf16_rne(gs[r])
            assert np.array_equal(u16(shard_g[r]), g16), f"bf16 shard grad rank {r} step {t}"
            p, m, v = O.adamw_update(O.bf16_to_f32(g16), st.master[r], st.m[r], st.v[r], sc)
            st.master[r], st.m[r], st.v[r] = p, m, v
            st.sparam[r] = O.cast_bf16(p)
    for r in range(nd):
        assert np.array_equal(bits(f32(e.master[r])), bits(st.master[r]))
        assert np.array_equal(u16(e.sparam[r]), st.sparam[r])


def test_reduce_scatter_worked_example_on_device(dev):
    """The pages' example: G0 = [2, 6], G1 = [4, 10] -> rank 0 [3], rank 1 [8]."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "reduce_scatter_example.json")))
    plan = zero3.Plan([2], None, 2, threshold=0)
    G = [torch.tensor(x, dtype=torch.bfloat16, device=dev) for x in g["local_grads"]]
    out = [torch.zeros(1, dtype=torch.float32, device=dev) for _ in range(2)]
    zero3.zero3_reduce_scatter(plan, [x.data_ptr() for x in G], 0, 0, 2,
                               [o.data_ptr() for o in out], zero3.F32, 0)
    torch.cuda.synchronize()
    assert [o.item() for o in out] == [float(v[0]) for v in g["reduce_scatter"]]


# ---------------------------------------------------------------- fetch + state machine
@pytest.mark.parametrize("wname", ["toy", "mini4", "ragged7"])
def test_fetch_submodule_matches_oracle(dev, wname):
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = {"toy": W.toy_mlp, "mini4": lambda: W.mini_gpt(4), "ragged7": lambda: W.ragged_small(7)}[wname]()
    plan, st, full, ps = oracle_run(w, 2)
    e = run_device(w, 2)
    for k in range(plan.n_submodules):
        e.fetch(k)
        assert zero3.zero3_submodule_status(e.plan, k) in (zero3.INFLIGHT, zero3.AVAILABLE)
        zero3.zero3_submodule_wait(e.plan, k)
        assert zero3.zero3_submodule_status(e.plan, k) == zero3.AVAILABLE
        n = plan.submodule_numel(k)
        ref = O.fetch_submodule(plan, k, st.sparam, ps.param)
        assert np.array_equal(u16(e.out)[:n], ref), f"submodule {k}"
        e.release(k)
        assert zero3.zero3_submodule_status(e.plan, k) == zero3.NOT_AVAILABLE


def test_fetch_state_machine_refcount(dev):
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.toy_mlp()
    e = make_emu(w)
    other = torch.empty_like(e.out)
    e.fetch(0)
    e.fetch(0)  # second reference, no new gather
    with pytest.raises(zero3.Zero3Error) as exc:
        zero3.zero3_fetch_submodule(e.plan, 0, e.ptrs(e.sparam), e.pparam.data_ptr(),
                                    other.data_ptr(), e.sid)
    assert exc.value.status == zero3.ESTATE
    zero3.zero3_sync(e.sid)
    assert zero3.zero3_submodule_status(e.plan, 0) == zero3.AVAILABLE
    e.release(0)
    assert zero3.zero3_submodule_status(e.plan, 0) == zero3.AVAILABLE
    e.release(0)
    assert zero3.zero3_submodule_status(e.plan, 0) == zero3.NOT_AVAILABLE
    with pytest.raises(zero3.Zero3Error) as exc:
        e.release(0)
    assert exc.value.status == zero3.ESTATE
    # after release the submodule can be gathered into another buffer
    zero3.zero3_fetch_submodule(e.plan, 0, e.ptrs(e.sparam), e.pparam.data_ptr(),
                                other.data_ptr(), e.sid)
    zero3.zero3_submodule_wait(e.plan, 0)
    n = e.plan.submodule(0)[1]
    assert torch.equal(other[:n].view(torch.int16), e.out[:n].view(torch.int16))
    e.release(0)


# ---------------------------------------------------------------- faults confined
def test_nan_gradient_stays_in_its_element(dev):
    """A NaN in one rank's gradient poisons only that element's outputs."""
    w = W.mini_gpt(4)
    e = make_emu(w)
    e.fill_grads(1)
    f = 12345
    e.grads[0][2][f] = float("nan")
    e.step(1)
    torch.cuda.synchronize()
    r, i = f // e.S, f % e.S
    master = f32(e.master[r])
    assert np.isnan(master[i])
    assert np.isnan(master).sum() == 1
    assert sum(int(np.isnan(f32(e.master[q])).sum()) for q in range(4)) == 1
    full = O.bf16_to_f32(u16(e.full))
    assert np.isnan(full[f]) and np.isnan(full).sum() == 1


def test_launch_after_bad_arguments_leaves_state_untouched(dev):
    """An invalid call launches nothing."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.toy_mlp()
    e = make_emu(w)
    e.fill_grads(1)
    before = f32(e.master[0]).copy()
    bad = e.ptrs(e.grads[0])
    bad[1] = 0
    with pytest.raises(zero3.Zero3Error):
        zero3.zero3_step(e.plan, e.hp, 1, bad, 0, e.ptrs(e.master), e.ptrs(e.m), e.ptrs(e.v),
                         e.ptrs(e.sparam), e.full.data_ptr(), e.persist, 0, e.psi_pad, e.sid)
    torch.cuda.synchronize()
    assert np.array_equal(bits(f32(e.master[0])), bits(before))


# ---------------------------------------------------------------- ZeRO-1/2 step
@pytest.mark.parametrize("nd", [2, 4, 7, 8])
def test_stage12_step_matches_oracle(dev, nd):
    """Every rank's full bf16 parameter copy and every fp32 shard after 3
    ZeRO-1/2 steps equal the oracle's replicated step, bit for bit."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    from tests._oracle_runs import host_master
    w = W.mini_gpt(nd)
    w.threshold = 0
    plan = O.partition(w.numels, w.submodule_of, nd, 0, w.bucket)
    assert plan.psi_s == 0
    e = make_emu(w)
    params = [e.full.clone() for _ in range(nd)]
    mf, mp = host_master(w, plan)
    st, full, _ = O.init_state(plan, mf, mp)
    ref = [full.copy() for _ in range(nd)]
    for t in range(1, 4):
        e.fill_grads(t)
        zero3.zero3_step_stage12(e.plan, e.hp, t, e.ptrs(e.grads[0]), 0, e.ptrs(e.master),
                                 e.ptrs(e.m), e.ptrs(e.v), [x.data_ptr() for x in params], 0,
                                 e.psi_pad, e.sid)
        O.replicated_step(plan, w.hparams, t, host_grads(w, plan, t), st, ref)
    torch.cuda.synchronize()
    for q in range(nd):
        assert np.array_equal(u16(params[q]), ref[q]), q
        assert np.array_equal(bits(f32(e.master[q])), bits(st.master[q]))
        assert np.array_equal(bits(f32(e.m[q])), bits(st.m[q]))
        assert np.array_equal(bits(f32(e.v[q])), bits(st.v[q]))


# ---------------------------------------------------------------- degenerate plans
def test_all_persistent_plan(dev):
    """Every tensor below the threshold: no flat range at all (psi_pad = 0),
    zero3_step over the empty range still updates the persistent group."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.toy_mlp()
    w.threshold = 10 ** 7
    plan, st, full, ps = oracle_run(w, 3)
    assert plan.psi_pad == 0 and plan.psi_s == w.psi
    e = make_emu(w)
    for t in range(1, 4):
        e.fill_grads(t)
        zero3.zero3_step(e.plan, e.hp, t, e.ptrs(e.pgrads), 0, [0] * 2, [0] * 2, [0] * 2,
                         [0] * 2, 0, e.persist, 0, 0, e.sid)
    torch.cuda.synchronize()
    assert np.array_equal(bits(f32(e.pmaster)), bits(ps.master))
    assert np.array_equal(u16(e.pparam), ps.param)
    e.fetch(0)
    torch.cuda.synchronize()
    assert np.array_equal(u16(e.out)[:plan.submodule_numel(0)],
                          O.fetch_submodule(plan, 0, st.sparam, ps.param))
    e.release(0)


def test_zero_size_tensors(dev):
    """Zero-element tensors anywhere in the list (persistent by the strict
    threshold) and a submodule made only of them: planner, step and fetch."""
    numels = [0, 300_000, 0, 5, 0, 200_001, 0]
    subs = [0, 0, 1, 1, 2, 3, 3]
    w = W.Workload("zeros", numels, subs, n_ranks=3, steps=3, seed=11)
    plan, st, full, ps = oracle_run(w, 3)
    e = run_device(w, 3)
    compare_all(e, plan, st, full, ps)
    from zero_sharded_optimizer_shard_gb300 import zero3
    e.full.zero_()
    zero3.zero3_allgather(e.plan, e.ptrs(e.sparam), e.full.data_ptr(), 0, e.psi_pad, e.sid)
    torch.cuda.synchronize()
    assert np.array_equal(u16(e.full), O.allgather(plan, st.sparam)), "unfused all-gather"
    for k in range(plan.n_submodules):
        e.fetch(k)
        torch.cuda.synchronize()
        n = plan.submodule_numel(k)
        assert np.array_equal(u16(e.out)[:n], O.fetch_submodule(plan, k, st.sparam, ps.param))
        e.release(k)
    # every submodule in one call, the empty one (only zero-size tensors) included
    ks = list(range(plan.n_submodules))
    outs = e.fetch_many(ks)
    torch.cuda.synchronize()
    for k, o in zip(ks, outs):
        n = plan.submodule_numel(k)
        off = (o - e.arena.data_ptr()) // 2
        assert np.array_equal(u16(e.arena)[off:off + n],
                              O.fetch_submodule(plan, k, st.sparam, ps.param)), k
        assert zero3.zero3_submodule_status(e.plan, k) != zero3.NOT_AVAILABLE
        e.release(k)


# ---------------------------------------------------------------- every phase
def all_phase_workload():
    """Two partitioned tensors and two persistent ones; the shard length is
    odd at N_d = 8, so rank r's shard starts at element phase (r * S) mod 8
    and the eight ranks take every phase 0..7 once (gradient and all-gather
    streams alike)."""
    return W.Workload("all_phases_nd8", [100_003, 160_005, 17, 99_999], [0, 1, 1, 2],
                      n_ranks=8, steps=3, seed=21)


def test_every_phase_fused_bucketed_and_fetch(dev):
    """Vector chunks read phased gradients as two aligned blocks, full warps
    store the phased all-gather cooperatively, span edges take the narrow
    paths: all bit-exact at every phase.  An odd bucket size shifts the
    gradient phases against the all-gather phases."""
    w = all_phase_workload()
    plan, st, full, ps = oracle_run(w, 3)
    assert plan.shard_len % 2 == 1
    assert sorted((r * plan.shard_len) % 8 for r in range(8)) == list(range(8))
    e = run_device(w, 3)
    compare_all(e, plan, st, full, ps)
    from zero_sharded_optimizer_shard_gb300 import zero3
    e.full.zero_()
    zero3.zero3_allgather(e.plan, e.ptrs(e.sparam), e.full.data_ptr(), 0, e.psi_pad, e.sid)
    torch.cuda.synchronize()
    assert np.array_equal(u16(e.full), O.allgather(plan, st.sparam)), "unfused all-gather"
    for k in range(plan.n_submodules):
        e.fetch(k)
        torch.cuda.synchronize()
        n = plan.submodule_numel(k)
        assert np.array_equal(u16(e.out)[:n], O.fetch_submodule(plan, k, st.sparam, ps.param)), k
        e.release(k)
    wb = all_phase_workload()
    wb.bucket = 7_919
    eb = run_device(wb, 3, bucketed=True)
    assert len(eb.chunks) > 8
    compare_all(eb, plan, st, full, ps)


def test_every_phase_stage12(dev):
    """The ZeRO-1/2 step writes all N_d full copies through the shared
    cooperative block at every phase."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    from tests._oracle_runs import host_master
    w = all_phase_workload()
    w.threshold = 0
    nd = w.n_ranks
    plan = O.partition(w.numels, w.submodule_of, nd, 0, w.bucket)
    assert plan.psi_s == 0 and plan.shard_len % 2 == 1
    e = make_emu(w)
    params = [e.full.clone() for _ in range(nd)]
    mf, mp = host_master(w, plan)
    st, full, _ = O.init_state(plan, mf, mp)
    ref = [full.copy() for _ in range(nd)]
    for t in range(1, 4):
        e.fill_grads(t)
        zero3.zero3_step_stage12(e.plan, e.hp, t, e.ptrs(e.grads[0]), 0, e.ptrs(e.master),
                                 e.ptrs(e.m), e.ptrs(e.v), [x.data_ptr() for x in params], 0,
                                 e.psi_pad, e.sid)
        O.replicated_step(plan, w.hparams, t, host_grads(w, plan, t), st, ref)
    torch.cuda.synchronize()
    for q in range(nd):
        assert np.array_equal(u16(params[q]), ref[q]), q
        assert np.array_equal(bits(f32(e.master[q])), bits(st.master[q])), q
