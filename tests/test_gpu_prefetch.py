"""The prefetching coordinator through the C ABI: gathered contents against
the oracle at every fetch of two forward/backward steps, with the prefetch
and compute streams deliberately delayed so that a missing wait would expose
stale or overwritten data; reuse at the forward/backward turn, recorded
order, departures from the order, tight arenas and state errors."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from tests._oracle_runs import host_grads, host_master, host_pgrads, u16  # noqa: E402
from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


def fwd_bwd(n):
    return list(range(n)) + list(reversed(range(n)))


def run(w, steps, order_of_step, arena_mult=3.0, bucket=10**9, reuse=10**9, trace="given",
        delay=True):
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    compute = torch.cuda.Stream()
    prefetch = torch.cuda.Stream()
    e = Emulation(w, stream=compute)
    with torch.cuda.stream(compute):
        e.init_params()
    plan = e.plan
    n_sub = plan.info.n_submodules
    sizes = [plan.submodule(k)[1] for k in range(n_sub)]
    arena_elems = (int(max(sizes) * arena_mult) + 7) // 8 * 8
    arena = torch.empty(arena_elems, dtype=torch.bfloat16, device="cuda")
    tr = fwd_bwd(n_sub) if trace == "given" else []
    co = zero3.Coordinator(plan, tr, e.ptrs(e.sparam), e.pparam.data_ptr(), arena.data_ptr(),
                           arena_elems, prefetch_bucket_size=bucket,
                           max_live_parameters=arena_elems, max_reuse_distance=reuse,
                           compute_stream=compute.cuda_stream, prefetch_stream=prefetch.cuda_stream)
    seen = []  # (step, k, snapshot)
    for t in range(1, steps + 1):
        with torch.cuda.stream(compute):
            e.fill_grads(t)
        for k in order_of_step(t, n_sub):
            if delay:
                with torch.cuda.stream(prefetch):
                    torch.cuda._sleep(200_000)
            ptr = co.fetch(k)
            with torch.cuda.stream(compute):
                if delay:
                    torch.cuda._sleep(100_000)
                n = sizes[k]
                off = (ptr - arena.data_ptr()) // 2
                assert 0 <= off and off + n <= arena_elems
                seen.append((t, k, arena[off:off + n].clone()))
            co.release(k)
        with torch.cuda.stream(compute):
            e.step(t)
        co.next_step()
    torch.cuda.synchronize()
    return e, co, seen


def oracle_params_by_step(w, steps):
    """bf16 shards and persistent params before each step's update."""
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    mf, mp = host_master(w, plan)
    st, full, ps = O.init_state(plan, mf, mp)
    before = {}
    for t in range(1, steps + 1):
        before[t] = ([x.copy() for x in st.sparam], ps.param.copy())
        O.sharded_step(plan, w.hparams, t, host_grads(w, plan, t), st, full)
        O.persistent_step(plan, w.hparams, t, host_pgrads(w, plan, t), ps, replicas=1)
    return plan, before


def check(seen, plan, before):
    for t, k, snap in seen:
        sp, pp = before[t]
        want = O.fetch_submodule(plan, k, sp, pp)
        assert np.array_equal(u16(snap), want), (t, k)


@pytest.mark.parametrize("arena_mult", [1.0, 1.5, 3.0])
def test_prefetched_contents_match_oracle(arena_mult):
    w = W.mini_gpt(4)
    e, co, seen = run(w, 2, lambda t, n: fwd_bwd(n), arena_mult=arena_mult)
    plan, before = oracle_params_by_step(w, 2)
    check(seen, plan, before)
    s = co.stats()
    assert s["steps"] == 2 and s["trace_misses"] == 0
    assert s["peak_live_elems"] <= int(max(plan.submodule_numel(k) for k in plan.submodules) * arena_mult)
    if arena_mult >= 3.0:
        assert s["prefetch_hits"] > 0
        # the last block is fetched at the end of forward and again at the
        # start of backward: kept (reuse distance 0) instead of re-gathered
        assert s["reuse_hits"] >= 2


def test_recorded_order_and_departures():
    """No trace given: the first step records the order (no prefetch), the
    second step prefetches; a third step in another order departs from it and
    stays correct."""
    w = W.mini_gpt(3)

    def order(t, n):
        return fwd_bwd(n) if t < 3 else list(range(n)) + list(range(n))
    e, co, seen = run(w, 3, order, trace="record")
    plan, before = oracle_params_by_step(w, 3)
    check(seen, plan, before)
    s = co.stats()
    assert s["prefetched"] > 0 and s["trace_misses"] >= 1


def test_no_prefetch_and_no_reuse_still_correct():
    w = W.ragged_small(7)
    e, co, seen = run(w, 2, lambda t, n: fwd_bwd(n), bucket=0, reuse=0, arena_mult=1.0)
    plan, before = oracle_params_by_step(w, 2)
    check(seen, plan, before)
    s = co.stats()
    # distance 0: only the last submodule at the forward/backward turn is
    # kept (nothing is fetched between its release and its next use)
    assert s["prefetched"] == 0 and s["reuse_hits"] == 2
    assert s["gathers"] == 2 * (2 * plan.n_submodules - 1)


def test_state_errors():
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    w = W.toy_mlp()
    compute, prefetch = torch.cuda.Stream(), torch.cuda.Stream()
    e = Emulation(w, stream=compute)
    e.init_params()
    n = max(e.plan.submodule(k)[1] for k in range(e.plan.info.n_submodules))
    n = (n + 7) // 8 * 8
    arena = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    co = zero3.Coordinator(e.plan, [0, 1, 2], e.ptrs(e.sparam), e.pparam.data_ptr(),
                           arena.data_ptr(), n, compute_stream=compute.cuda_stream,
                           prefetch_stream=prefetch.cuda_stream)
    with pytest.raises(zero3.Zero3Error) as exc:
        co.release(0)
    assert exc.value.status == zero3.ESTATE
    co.fetch(0)
    with pytest.raises(zero3.Zero3Error) as exc:
        co.next_step()
    assert exc.value.status == zero3.ESTATE
    # the arena holds one submodule: another fetch while 0 is held has no room
    with pytest.raises(zero3.Zero3Error) as exc:
        co.fetch(1)
    assert exc.value.status == zero3.ENOMEM
    torch.cuda.synchronize()


def test_odd_sized_submodules_share_the_arena():
    """Ragged submodule sizes with room for several copies at once: every
    copy must start 16-byte aligned inside the arena (ranges are rounded to
    8 elements) and hold the oracle's contents."""
    w = W.ragged_small(7)
    e, co, seen = run(w, 2, lambda t, n: fwd_bwd(n), arena_mult=4.0, delay=False)
    plan, before = oracle_params_by_step(w, 2)
    check(seen, plan, before)
    assert co.stats()["prefetch_hits"] > 0


def test_prefetch_batches_many_small_submodules():
    """Ragged list, arena for the whole model: the prefetch window goes out
    as a few batched gathers (far fewer launches than submodules gathered),
    the compute stream waits once per batch, and every copy still equals the
    oracle's gather of the parameters before that step."""
    w = W.ragged_small(7)
    plan0 = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    total = sum(plan0.submodule_numel(k) for k in plan0.submodules)
    big = max(plan0.submodule_numel(k) for k in plan0.submodules)
    e, co, seen = run(w, 2, lambda t, n: fwd_bwd(n), arena_mult=2.2 * total / big, delay=False)
    plan, before = oracle_params_by_step(w, 2)
    check(seen, plan, before)
    s = co.stats()
    assert s["trace_misses"] == 0 and s["prefetched"] > 0
    assert s["gather_launches"] * 10 < s["gathers"], s
    assert s["gather_calls"] * 10 < s["gathers"], s
    fetches = 2 * 2 * plan.n_submodules
    assert s["compute_waits"] * 10 < fetches, s
