"""Stream order between this library's kernels and other kernels on the same
stream.  Every kernel of the library is launched so that it may be scheduled
while the previous kernel of its stream drains, and waits for the previous
grids (and their writes) before its first memory access.  These tests put
torch kernels that rewrite a call's inputs, and torch kernels that read its
outputs, directly before and after the library's launches on one stream,
without any synchronisation, and check every intermediate result against the
oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from tests._oracle_runs import u16  # noqa: E402
from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda:0")


def pattern(i, r):
    """A bf16 bit pattern distinct per round i and rank r (1.0 .. 1.98)."""
    return 0x3F80 + ((7 * i + r) % 127)


def emu(w):
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    s = torch.cuda.Stream()
    e = Emulation(w, stream=s)
    with torch.cuda.stream(s):
        e.init_params()
    torch.cuda.synchronize()
    return e, s


@pytest.mark.parametrize("wname", ["mini4", "ragged7"])
def test_fetch_sees_preceding_writes_and_feeds_following_reads(dev, wname):
    w = {"mini4": lambda: W.mini_gpt(4), "ragged7": lambda: W.ragged_small(7)}[wname]()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e, s = emu(w)
    n_sub = plan.n_submodules
    rounds = 3 * n_sub
    snaps = []
    with torch.cuda.stream(s):
        for i in range(rounds):
            k = i % n_sub
            for r in range(plan.n_ranks):
                e.sparam[r].view(torch.int16).fill_(pattern(i, r))
            e.pparam.view(torch.int16).fill_(pattern(i, 99))
            e.fetch(k)
            n = plan.submodule_numel(k)
            snaps.append((i, k, e.out[:n].clone()))
            e.out.view(torch.int16).fill_(0x7FC1)     # overwritten by the next fetch
            e.release(k)
    torch.cuda.synchronize()
    for i, k, got in snaps:
        sp = [np.full(plan.shard_len, pattern(i, r), np.uint16) for r in range(plan.n_ranks)]
        pp = np.full(plan.psi_s, pattern(i, 99), np.uint16)
        ref = O.fetch_submodule(plan, k, sp, pp)
        assert np.array_equal(u16(got), ref), f"round {i}, submodule {k}"


def test_allgather_between_torch_kernels(dev):
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.mini_gpt(4)
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e, s = emu(w)
    snaps = []
    with torch.cuda.stream(s):
        for i in range(20):
            for r in range(plan.n_ranks):
                e.sparam[r].view(torch.int16).fill_(pattern(i, r))
            zero3.zero3_allgather(e.plan, e.ptrs(e.sparam), e.full.data_ptr(), 0, e.psi_pad, e.sid)
            snaps.append((i, e.full.clone()))
            e.full.view(torch.int16).fill_(0x7FC1)
    torch.cuda.synchronize()
    for i, got in snaps:
        sp = [np.full(plan.shard_len, pattern(i, r), np.uint16) for r in range(plan.n_ranks)]
        assert np.array_equal(u16(got), O.allgather(plan, sp)), f"round {i}"


def test_step_chain_with_torch_kernels_between(dev):
    """Ten fused steps, each fed by gradients that torch copies into place
    right before the launch, and each followed by torch copies of the state:
    every snapshot equals the oracle after that step."""
    from tests._oracle_runs import host_grads, host_master, host_pgrads
    w = W.mini_gpt(4)
    T = 10
    e, s = emu(w)
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    host = [(host_grads(w, plan, t), host_pgrads(w, plan, t)) for t in range(1, T + 1)]
    staged = [([torch.from_numpy(g.view(np.int16)).to(dev) for g in G],
               [torch.from_numpy(g.view(np.int16)).to(dev) for g in PG]) for G, PG in host]
    torch.cuda.synchronize()
    snaps = []
    with torch.cuda.stream(s):
        for t in range(1, T + 1):
            G, PG = staged[t - 1]
            for q in range(plan.n_ranks):
                e.grads[0][q].view(torch.int16).copy_(G[q])
                e.pgrads[q].view(torch.int16).copy_(PG[q])
            e.step(t)
            snaps.append((e.master[0].clone(), e.full.clone(), e.pmaster.clone()))
    torch.cuda.synchronize()
    mf, mp = host_master(w, plan)
    st, full, ps = O.init_state(plan, mf, mp)
    for t in range(1, T + 1):
        G, PG = host[t - 1]
        O.sharded_step(plan, w.hparams, t, G, st, full)
        O.persistent_step(plan, w.hparams, t, PG, ps)
        m0, f, pm = snaps[t - 1]
        assert np.array_equal(m0.cpu().numpy().view(np.uint32), st.master[0].view(np.uint32)), t
        assert np.array_equal(u16(f), full), t
        assert np.array_equal(pm.cpu().numpy().view(np.uint32), ps.master.view(np.uint32)), t


def test_fused_step_replays_from_a_cuda_graph(dev):
    """The fused step (flat range + persistent group) captured once in a CUDA
    graph and replayed three times equals three oracle steps with the same
    step count and gradients: the launches are capturable, and the
    programmatic ordering holds between replays."""
    from tests._oracle_runs import host_grads, host_master, host_pgrads
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.mini_gpt(4)
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e, s = emu(w)
    with torch.cuda.stream(s):
        e.fill_grads(1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        e.step(1)
        zero3.zero3_allgather(e.plan, e.ptrs(e.sparam), e.full.data_ptr(), 0, e.psi_pad, e.sid)
    torch.cuda.synchronize()
    snaps = []
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
            snaps.append((e.master[1].clone(), e.v[1].clone(), e.full.clone(), e.pparam.clone()))
    torch.cuda.synchronize()
    mf, mp = host_master(w, plan)
    st, full, ps = O.init_state(plan, mf, mp)
    G, PG = host_grads(w, plan, 1), host_pgrads(w, plan, 1)
    for k in range(3):
        O.sharded_step(plan, w.hparams, 1, G, st, full)
        O.persistent_step(plan, w.hparams, 1, PG, ps)
        m1, v1, f, pp = snaps[k]
        assert np.array_equal(m1.cpu().numpy().view(np.uint32), st.master[1].view(np.uint32)), k
        assert np.array_equal(v1.cpu().numpy().view(np.uint32), st.v[1].view(np.uint32)), k
        assert np.array_equal(u16(f), O.allgather(plan, st.sparam)), k
        assert np.array_equal(u16(pp), ps.param), k


@pytest.mark.parametrize("bits", [8, 4])
def test_qwz_step_and_dequantizing_gather_replay_from_a_cuda_graph(dev, bits):
    """The qwZ step and the dequantizing all-gather (a piece launch whose
    sources sit at nonzero phases: the ragged list at N_d = 7) captured once
    in a CUDA graph and replayed three times equal three oracle steps with the
    same step count and gradients, codes and gathered bf16 bit for bit."""
    from tests._oracle_runs import host_grads, host_master
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = W.ragged_small(7)
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e, s = emu(w)
    assert e.S % 8 != 0  # the shards start at nonzero phases in the flat buffer
    nb = -(-e.S // 256)
    codes = [torch.zeros(max(e.S, 16), dtype=torch.int8, device=dev) for _ in range(e.nd)]
    scales = [torch.zeros(max(nb, 4), dtype=torch.float32, device=dev) for _ in range(e.nd)]
    with torch.cuda.stream(s):
        e.fill_grads(1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        zero3.zero3_step_qwz(e.plan, e.hp, 1, e.ptrs(e.grads[0]), 0, e.ptrs(e.master), e.ptrs(e.m),
                             e.ptrs(e.v), e.ptrs(e.sparam), e.ptrs(codes), e.ptrs(scales), None,
                             0, e.psi_pad, e.sid, bits=bits)
        zero3.zero3_allgather_qwz(e.plan, e.ptrs(codes), e.ptrs(scales), e.full.data_ptr(), 0,
                                  e.psi_pad, e.sid, bits=bits)
    torch.cuda.synchronize()
    snaps = []
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
            snaps.append(([m.clone() for m in e.master], e.full.clone()))
    torch.cuda.synchronize()
    mf, mp = host_master(w, plan)
    st, full, _ = O.init_state(plan, mf, mp)
    G = host_grads(w, plan, 1)
    for k in range(3):
        O.sharded_step(plan, w.hparams, 1, G, st, full)
        q = [O.qwz_quantize(st.sparam[r], bits=bits) for r in range(w.n_ranks)]
        want = O.qwz_allgather(plan, [c for c, _ in q], [sc for _, sc in q])
        masters, f = snaps[k]
        for r in range(w.n_ranks):
            assert np.array_equal(masters[r].cpu().numpy().view(np.uint32),
                                  st.master[r].view(np.uint32)), (k, r)
        assert np.array_equal(u16(f), want), k
