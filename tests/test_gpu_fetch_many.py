"""zero3_fetch_submodules: several submodules gathered by shared launches,
through the C ABI, against the oracle's per-submodule gather, and the
ZeroParamStatus transitions it makes for every submodule it lists."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from tests._oracle_runs import oracle_run, u16  # noqa: E402
from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda:0")


def run_device(w, T):
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    e = Emulation(w)
    e.init_params()
    for t in range(1, T + 1):
        e.fill_grads(t)
        e.step(t)
    torch.cuda.synchronize()
    return e


def many_pieces():
    """1500 tensors of 1 to 3000 elements (threshold 1000, N_d = 7): about
    as many pieces as tensors, so one call over every submodule needs
    several launches of 512 pieces, and most pieces are shorter than one
    warp's 1024 elements."""
    w = W.ragged(n_tensors=1500, n_ranks=7, small_hi=1e3, big_lo=1e3, big_hi=3e3)
    w.threshold = 1000
    w.name = "many_pieces_nd7"
    return w


def all_phases():
    return W.Workload("all_phases_nd8", [100_003, 160_005, 17, 99_999, 3, 250_007],
                      [0, 1, 1, 2, 3, 3], n_ranks=8, steps=2, seed=21)


WORKLOADS = {"toy": W.toy_mlp, "mini4": lambda: W.mini_gpt(4),
             "ragged7": lambda: W.ragged_small(7), "many": many_pieces, "phases": all_phases}


def check(e, plan, st, ps, ks, outs):
    for k, o in zip(ks, outs):
        n = plan.submodule_numel(k)
        got = u16(e.arena)[(o - e.arena.data_ptr()) // 2:][:n]
        assert np.array_equal(got, O.fetch_submodule(plan, k, st.sparam, ps.param)), k


@pytest.mark.parametrize("wname", sorted(WORKLOADS))
def test_fetch_submodules_matches_oracle(dev, wname):
    """Every submodule in one call, then buckets of a few submodules, then
    the bucketed forward/backward pass of the step: each gathered buffer
    equals the oracle's gather of that submodule, bit for bit."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = WORKLOADS[wname]()
    plan, st, full, ps = oracle_run(w, 2)
    e = run_device(w, 2)
    n = plan.n_submodules
    ks = list(range(n))
    if wname == "many":
        pieces = sum(1 if e.plan.tensor(t).persistent else e.plan.tensor(t).n_segments
                     for t in range(len(w.numels)) if w.numels[t] > 0)
        assert pieces > 2 * 512  # several launches in one call
    e.arena = None
    outs = e.fetch_many(ks)
    for k in ks:
        zero3.zero3_submodule_wait(e.plan, k)
        assert zero3.zero3_submodule_status(e.plan, k) == zero3.AVAILABLE
    check(e, plan, st, ps, ks, outs)
    for k in ks:
        e.release(k)
        assert zero3.zero3_submodule_status(e.plan, k) == zero3.NOT_AVAILABLE
    # buckets of consecutive submodules, in reverse order (backward pass)
    total = sum(plan.submodule_numel(k) for k in ks)
    for g in reversed(e.gather_buckets(max(1, total // 5))):
        g = list(reversed(g))
        e.arena.view(torch.int16).fill_(-1)
        outs = e.fetch_many(g)
        torch.cuda.synchronize()
        check(e, plan, st, ps, g, outs)
        for k in g:
            e.release(k)
    e.forward_backward_gathers(bucket=max(1, total // 3))
    torch.cuda.synchronize()
    for k in ks:
        assert zero3.zero3_submodule_status(e.plan, k) == zero3.NOT_AVAILABLE


def test_fetch_submodules_state_machine(dev):
    """References and outputs follow n single fetches in list order; a call
    with a conflicting output changes nothing and launches nothing."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.mini_gpt(4)
    plan, st, full, ps = oracle_run(w, 1)
    e = run_device(w, 1)
    P, pp = e.ptrs(e.sparam), e.pparam.data_ptr()
    n = plan.n_submodules
    assert n >= 3
    outs = e.bucket_outputs([0, 1, 2])
    # 1 gathered alone first, then listed again with its own output
    zero3.zero3_fetch_submodule(e.plan, 1, P, pp, outs[1], e.sid)
    e.arena.view(torch.int16).fill_(0)
    torch.cuda.synchronize()
    arena_before = e.arena.clone()
    # a conflicting output for 1 (already fetched): ESTATE, nothing gathered
    with pytest.raises(zero3.Zero3Error) as exc:
        zero3.zero3_fetch_submodules(e.plan, [0, 1, 2], P, pp, [outs[0], outs[0], outs[2]], e.sid)
    assert exc.value.status == zero3.ESTATE
    # a submodule listed twice with two outputs: ESTATE, nothing gathered
    with pytest.raises(zero3.Zero3Error) as exc:
        zero3.zero3_fetch_submodules(e.plan, [0, 2, 0], P, pp, [outs[0], outs[2], outs[2]], e.sid)
    assert exc.value.status == zero3.ESTATE
    # bad id and misaligned output: EINVAL
    with pytest.raises(zero3.Zero3Error) as exc:
        zero3.zero3_fetch_submodules(e.plan, [0, n], P, pp, [outs[0], outs[0]], e.sid)
    assert exc.value.status == zero3.EINVAL
    with pytest.raises(zero3.Zero3Error) as exc:
        zero3.zero3_fetch_submodules(e.plan, [0], P, pp, [outs[0] + 2], e.sid)
    assert exc.value.status == zero3.EINVAL
    torch.cuda.synchronize()
    assert torch.equal(e.arena, arena_before)
    for k in (0, 2):
        assert zero3.zero3_submodule_status(e.plan, k) == zero3.NOT_AVAILABLE
    # the valid call: 0 twice, 1 already fetched (same output), 2 once
    zero3.zero3_fetch_submodules(e.plan, [0, 1, 2, 0], P, pp, [outs[0], outs[1], outs[2], outs[0]],
                                 e.sid)
    torch.cuda.synchronize()
    check(e, plan, st, ps, [0, 2], [outs[0], outs[2]])  # 1 was gathered before the fill
    refs = {0: 2, 1: 2, 2: 1}
    for k, r in refs.items():
        for i in range(r):
            assert zero3.zero3_submodule_status(e.plan, k) != zero3.NOT_AVAILABLE
            e.release(k)
        assert zero3.zero3_submodule_status(e.plan, k) == zero3.NOT_AVAILABLE
    # an empty list does nothing
    zero3.zero3_fetch_submodules(e.plan, [], P, pp, [], e.sid)
