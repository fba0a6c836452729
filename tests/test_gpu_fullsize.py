"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark uses (bucketed gathers, the persistent group in the first fused
launch), on sampled outputs the oracle computes one by one (elementwise
independence of the update), plus the whole persistent group.

Sample: random flat indices plus every rank's first and last two local
indices, tensor boundaries and the padding."""
import gc

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from tests._oracle_runs import (assert_bf16_close, assert_f32_close, bits, f32,  # noqa: E402
                                host_master_persist, host_pgrads, sampled_oracle,
                                sampled_persistent_oracle, u16)
from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def sample_indices(plan, lo, hi, n, seed):
    rng = np.random.default_rng(seed)
    S = plan.shard_len
    idx = set(int(x) for x in rng.integers(lo, hi, n))
    for r in range(plan.n_ranks):
        for f in (r * S, r * S + 1, (r + 1) * S - 2, (r + 1) * S - 1):
            if lo <= f < hi:
                idx.add(f)
    for t in range(len(plan.numel)):
        if not plan.persistent[t]:
            for f in (plan.offset[t], plan.offset[t] + plan.numel[t] - 1):
                if lo <= f < hi:
                    idx.add(f)
    for f in range(plan.psi_p, plan.psi_pad):
        if lo <= f < hi:
            idx.add(f)
    return np.array(sorted(idx), np.int64)


def persistent_oracle(w, plan, T, grad_step=None):
    mp = host_master_persist(w, plan)
    ps = O.PersistState(mp.copy(), np.zeros_like(mp), np.zeros_like(mp), O.cast_bf16(mp))
    for t in range(1, T + 1):
        O.persistent_step(plan, w.hparams, t, host_pgrads(w, plan, t if grad_step is None else grad_step),
                          ps, replicas=2)
    return ps


def check_sample(e, plan, w, idx, T, grad_step=None):
    p, m, v, h = sampled_oracle(w, plan, idx, T, grad_step)
    S = plan.shard_len
    r = idx // S
    i = idx % S
    gm = np.empty(len(idx), np.float32)
    gmm = np.empty(len(idx), np.float32)
    gv = np.empty(len(idx), np.float32)
    gs = np.empty(len(idx), np.uint16)
    for q in np.unique(r):
        sel = r == q
        ii = torch.from_numpy(i[sel]).to(e.master[q].device)
        gm[sel] = f32(e.master[q][ii])
        gmm[sel] = f32(e.m[q][ii])
        gv[sel] = f32(e.v[q][ii])
        gs[sel] = u16(e.sparam[q][ii])
    gfull = u16(e.full[torch.from_numpy(idx).to(e.full.device)])
    for name, got, ref in (("master", gm, p), ("m", gmm, m), ("v", gv, v)):
        assert_f32_close(got, ref, what=name)
        assert np.array_equal(bits(got), bits(ref)), f"{name} not bit-exact"
    assert_bf16_close(gs, h, what="sparam")
    assert np.array_equal(gs, h) and np.array_equal(gfull, h)


def check_persistent(e, ps):
    for name, got, ref in (("pmaster", e.pmaster, ps.master), ("pm", e.pm, ps.m), ("pv", e.pv, ps.v)):
        g = f32(got)
        assert_f32_close(g, ref, what=name)
        assert np.array_equal(bits(g), bits(ref)), name
    assert np.array_equal(u16(e.pparam), ps.param)


def run(w, T, grad_step=None, **kw):
    """T steps as the benchmark runs them: the forward and backward gathers
    in all-gather buckets of the workload's size, then the fused step with the
    persistent group in its first launch."""
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    e = Emulation(w, **kw)
    e.init_params()
    for t in range(1, T + 1):
        if grad_step is None or t == 1:
            e.fill_grads(t if grad_step is None else grad_step)
        e.forward_backward_gathers(bucket=w.gather_bucket)
        e.step(t)
    torch.cuda.synchronize()
    return e


def check_fetch_many(e, plan, w, T, grad_step, groups, persist_values, state_ranks=None,
                     n=2000, seed=7):
    """zero3_fetch_submodules over the benchmark's all-gather buckets: each
    submodule's gathered buffer at sampled positions (and its ends) against
    the oracle's bf16 parameters of the same elements.  Ranks outside
    state_ranks hold their initial shards (cast from the initial masters);
    persist_values(pidx) gives the persistent group's bf16 values."""
    from zero_sharded_optimizer_shard_gb300 import synth
    from zero_sharded_optimizer_shard_gb300.workloads import STREAM_MASTER
    rng = np.random.default_rng(seed)
    S = plan.shard_len
    for ks in groups:
        outs = e.fetch_many(ks)
        torch.cuda.synchronize()
        base_ptr = e.arena.data_ptr()
        for k, o in zip(ks, outs):
            members = plan.submodules.get(k, [])
            pos, flat, pers = [], [], []
            base = 0
            for t in members:
                nt = plan.numel[t]
                if nt == 0:
                    continue
                js = np.unique(np.concatenate([rng.integers(0, nt, min(nt, n // len(members) + 1)),
                                               [0, nt - 1]]))
                for j in js:
                    pos.append(base + j)
                    flat.append(-1 if plan.persistent[t] else plan.offset[t] + j)
                    pers.append(plan.offset[t] + j if plan.persistent[t] else -1)
                base += nt
            if not pos:
                continue
            pos, flat, pers = np.array(pos), np.array(flat), np.array(pers)
            off = (o - base_ptr) // 2
            got = u16(e.arena[torch.from_numpy(off + pos).to(e.arena.device)])
            want = np.empty(len(pos), np.uint16)
            fsel = flat >= 0
            upd = fsel.copy()
            if state_ranks is not None:
                upd &= np.isin(flat // S, state_ranks)
            if upd.any():
                want[upd] = sampled_oracle(w, plan, flat[upd], T, grad_step)[3]
            init = fsel & ~upd
            if init.any():
                want[init] = O.bf16_rne(synth.normal_f32(w.seed, STREAM_MASTER, 0, 0, flat[init],
                                                         w.master_sigma))
            if (~fsel).any():
                want[~fsel] = persist_values(pers[~fsel])
            assert np.array_equal(got, want), f"submodule {k}"
        for k in ks:
            e.release(k)


def check_fetch(e, plan, w, T, grad_step, ks, ps, n=4000, seed=0):
    """Gathered submodule outputs at sampled positions against the oracle's
    bf16 parameters of the same flat / persistent elements."""
    rng = np.random.default_rng(seed)
    for k in ks:
        e.fetch(k)
        torch.cuda.synchronize()
        members = plan.submodules[k]
        pos, flat, pers = [], [], []
        base = 0
        for t in members:
            nt = plan.numel[t]
            js = np.unique(np.concatenate([rng.integers(0, nt, min(nt, n // len(members) + 1)),
                                           [0, nt - 1]]))
            for j in js:
                pos.append(base + j)
                if plan.persistent[t]:
                    flat.append(-1)
                    pers.append(plan.offset[t] + j)
                else:
                    flat.append(plan.offset[t] + j)
                    pers.append(-1)
            base += nt
        pos, flat, pers = np.array(pos), np.array(flat), np.array(pers)
        got = u16(e.out[torch.from_numpy(pos).to(e.out.device)])
        want = np.empty(len(pos), np.uint16)
        fsel = flat >= 0
        if fsel.any():
            want[fsel] = sampled_oracle(w, plan, flat[fsel], T, grad_step)[3]
        if (~fsel).any():
            want[~fsel] = ps.param[pers[~fsel]]
        assert np.array_equal(got, want), f"submodule {k}"
        e.release(k)


def test_gpt2_small_ten_steps():
    w = W.gpt2_small()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e = run(w, 10)
    check_sample(e, plan, w, sample_indices(plan, 0, plan.psi_pad, 150_000, 1), 10)
    ps = persistent_oracle(w, plan, 10)
    check_persistent(e, ps)
    check_fetch(e, plan, w, 10, None, [0, 5, plan.n_submodules - 1], ps)


def test_decoder_1p3b_bench_configuration():
    """The benchmark's workload and launch configuration: full emulation of
    N_d = 8 ranks, one fused launch over the whole flat range, gradients
    generated once and reused by every step."""
    w = W.decoder_1p3b()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    T = 3
    e = run(w, T, grad_step=1)
    check_sample(e, plan, w, sample_indices(plan, 0, plan.psi_pad, 120_000, 2), T, grad_step=1)
    ps = persistent_oracle(w, plan, T, grad_step=1)
    check_persistent(e, ps)
    check_fetch(e, plan, w, T, 1, [0, 12, plan.n_submodules - 1], ps)
    groups = e.gather_buckets(w.gather_bucket)
    assert len(groups) >= 2
    check_fetch_many(e, plan, w, T, 1, [groups[0], groups[-1]], lambda i: ps.param[i])


@pytest.mark.parametrize("nbits", [8, 4])
def test_decoder_1p3b_qwz_bench_configuration(nbits):
    """The qwZ benchmark's launch configuration at full size: the 1.3B list at
    N_d = 8, one quantizing fused step over the whole flat range, then the
    dequantizing all-gather, three steps on the same gradients.  Sampled
    256-element blocks (random ones and every rank's first and last, the
    last one partial where S is not a multiple of 256): the packed codes, the
    block scale and the gathered bf16 equal the oracle's quantization of the
    oracle's step there, bit for bit."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    w = W.decoder_1p3b()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e = Emulation(w, bucketed=False)
    e.init_params()
    e.fill_grads(1)
    S, nd, blk = e.S, e.nd, 256
    nb = -(-S // blk)
    codes = [torch.empty(-(-S * nbits // 8), dtype=torch.int8, device="cuda") for _ in range(nd)]
    scales = [torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(nd)]
    lo, hi = e.chunks[0]
    T = 3
    for t in range(1, T + 1):
        zero3.zero3_step_qwz(e.plan, e.hp, t, e.ptrs(e.grads[0]), lo, e.ptrs(e.master),
                             e.ptrs(e.m), e.ptrs(e.v), e.ptrs(e.sparam), e.ptrs(codes),
                             e.ptrs(scales), None, lo, hi, e.sid, bits=nbits)
        zero3.zero3_allgather_qwz(e.plan, e.ptrs(codes), e.ptrs(scales), e.full.data_ptr(), lo,
                                  hi, e.sid, bits=nbits)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11 + nbits)
    blocks = {(r, b) for r in range(nd) for b in (0, nb - 1)}
    blocks |= {(int(rng.integers(0, nd)), int(rng.integers(0, nb))) for _ in range(400)}
    blocks = sorted(blocks)
    spans = [(r, b, r * S + b * blk, r * S + min((b + 1) * blk, S)) for r, b in blocks]
    idx = np.concatenate([np.arange(f0, f1, dtype=np.int64) for _, _, f0, f1 in spans])
    _, _, _, h = sampled_oracle(w, plan, idx, T, grad_step=1)
    got_full = u16(e.full[torch.from_numpy(idx).to(e.full.device)])
    want_full = np.empty_like(h)
    pos = 0
    for r, b, f0, f1 in spans:
        n = f1 - f0
        c, sc = O.qwz_quantize(h[pos:pos + n], bits=nbits)
        want_full[pos:pos + n] = O.qwz_dequantize(c, sc)
        packed = O.qwz_pack(c, nbits)
        b0 = b * blk * nbits // 8
        got_codes = codes[r][b0:b0 + packed.size].cpu().numpy().view(np.uint8)
        assert np.array_equal(got_codes, packed), (r, b)
        assert np.array_equal(bits(f32(scales[r][b:b + 1])), bits(sc[:1])), (r, b)
        pos += n
    assert np.array_equal(got_full, want_full)


def test_decoder_1p3b_stage12_bench_configuration():
    """The ZeRO-1/2 benchmark's launch configuration at full size: the 1.3B
    list at N_d = 8, every rank holding full bf16 parameters, one fused launch
    over the whole flat range writing all eight copies, three steps on the
    same gradients.  Sampled flat indices (random, shard, tensor and padding
    edges): every rank's fp32 state and every rank's copy of the parameter
    equal the oracle's step there, bit for bit."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    w = W.decoder_1p3b()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e = Emulation(w, bucketed=False)
    e.init_params()
    e.fill_grads(1)
    params = [e.full.clone() for _ in range(w.n_ranks)]
    lo, hi = e.chunks[0]
    T = 3
    for t in range(1, T + 1):
        zero3.zero3_step_stage12(e.plan, e.hp, t, e.ptrs(e.grads[0]), lo, e.ptrs(e.master),
                                 e.ptrs(e.m), e.ptrs(e.v), [x.data_ptr() for x in params],
                                 lo, hi, e.sid)
    torch.cuda.synchronize()
    idx = sample_indices(plan, 0, plan.psi_pad, 60_000, 5)
    p, m, v, h = sampled_oracle(w, plan, idx, T, grad_step=1)
    S = plan.shard_len
    r, i = idx // S, idx % S
    for q in np.unique(r):
        sel = r == q
        ii = torch.from_numpy(i[sel]).to(e.master[q].device)
        for name, buf, ref in (("master", e.master[q], p), ("m", e.m[q], m), ("v", e.v[q], v)):
            assert np.array_equal(bits(f32(buf[ii])), bits(ref[sel])), (name, q)
    ti = torch.from_numpy(idx).to(params[0].device)
    for q in range(w.n_ranks):
        assert np.array_equal(u16(params[q][ti]), h), q


def test_decoder_1p3b_unfused_bench_configuration():
    """The unfused ablation's launch configuration at full size: the 1.3B
    list at N_d = 8, fp32 reduce-scatter into per-rank shard gradients, the
    AdamW launch, the all-gather launch, each over the whole flat range, two
    steps on the same gradients.  Sampled indices: states, shards and the
    gathered buffer equal the oracle's step, bit for bit (the fp32 unfused
    path computes exactly what the fused step computes)."""
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    w = W.decoder_1p3b()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e = Emulation(w, bucketed=False)
    e.init_params()
    e.fill_grads(1)
    sg = [torch.empty(e.S, dtype=torch.float32, device="cuda") for _ in range(e.nd)]
    lo, hi = e.chunks[0]
    T = 2
    for t in range(1, T + 1):
        zero3.zero3_reduce_scatter(e.plan, e.ptrs(e.grads[0]), lo, lo, hi, e.ptrs(sg), zero3.F32,
                                   e.sid)
        zero3.zero3_adamw_step(e.plan, e.hp, t, e.ptrs(sg), zero3.F32, e.ptrs(e.master),
                               e.ptrs(e.m), e.ptrs(e.v), e.ptrs(e.sparam), lo, hi, e.sid)
        zero3.zero3_allgather(e.plan, e.ptrs(e.sparam), e.full.data_ptr(), lo, hi, e.sid)
    torch.cuda.synchronize()
    check_sample(e, plan, w, sample_indices(plan, 0, plan.psi_pad, 60_000, 6), T, grad_step=1)


def test_decoder_1p3b_coordinator_bench_configuration():
    """The prefetching coordinator in its benchmark configuration at full
    size: the 1.3B list, the forward-then-backward trace over every
    submodule, an arena of three times the largest submodule, two steps'
    traces with the step boundary between them.  After every fetch, sampled
    positions of the gathered copy (and its ends) are read on the compute
    stream before the release; each equals the oracle's bf16 parameter of
    that element (the initial parameters: no optimizer step runs)."""
    from zero_sharded_optimizer_shard_gb300 import synth, zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    from zero_sharded_optimizer_shard_gb300.workloads import STREAM_MASTER
    w = W.decoder_1p3b()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    e = Emulation(w, bucketed=False)
    e.init_params()
    n_sub = e.plan.info.n_submodules
    sizes = [e.plan.submodule(k)[1] for k in range(n_sub)]
    trace = list(range(n_sub)) + list(reversed(range(n_sub)))
    arena_elems = (3 * max(sizes) + 7) // 8 * 8
    arena = torch.empty(arena_elems, dtype=torch.bfloat16, device="cuda")
    compute, prefetch = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    co = zero3.Coordinator(e.plan, trace, e.ptrs(e.sparam), e.pparam.data_ptr(), arena.data_ptr(),
                           arena_elems, prefetch_bucket_size=w.bucket,
                           max_live_parameters=arena_elems, max_reuse_distance=10**9,
                           compute_stream=compute.cuda_stream,
                           prefetch_stream=prefetch.cuda_stream)
    rng = np.random.default_rng(9)
    pers_init = O.cast_bf16(host_master_persist(w, plan))
    snaps = []
    for _ in range(2):
        for k in trace:
            members = [t for t in plan.submodules.get(k, []) if plan.numel[t] > 0]
            pos, want = [], []
            base = 0
            for t in members:
                nt = plan.numel[t]
                js = np.unique(np.concatenate([rng.integers(0, nt, 300), [0, nt - 1]]))
                pos.append(base + js)
                if plan.persistent[t]:
                    want.append(pers_init[plan.offset[t] + js])
                else:
                    want.append(O.bf16_rne(synth.normal_f32(w.seed, STREAM_MASTER, 0, 0,
                                                            plan.offset[t] + js, w.master_sigma)))
                base += nt
            ptr = co.fetch(k)
            if pos:
                pos = np.concatenate(pos)
                off = (ptr - arena.data_ptr()) // 2
                ti = torch.from_numpy(off + pos).to(arena.device)
                with torch.cuda.stream(compute):
                    snaps.append((k, arena[ti], np.concatenate(want)))
            co.release(k)
        co.next_step()
    torch.cuda.synchronize()
    stats = co.stats()
    del co
    assert stats["prefetched"] > 0
    for k, got, want in snaps:
        assert np.array_equal(u16(got), want), f"submodule {k}"


def test_llama_7b_rank0_view():
    """Rank 0's state only, gradients in 5e8-element bucket buffers (two
    launches per step), bf16 all-gather into the 6.7B-element full buffer."""
    w = W.llama_7b()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    T = 2
    e = run(w, T, state_ranks=[0], bucketed=True)
    assert len(e.chunks) == 2
    check_sample(e, plan, w, sample_indices(plan, 0, plan.shard_len, 100_000, 3), T)
    ps = persistent_oracle(w, plan, T)
    check_persistent(e, ps)
    # the bench's bucketed gathers: the first bucket (embeddings and the first
    # layer, mostly rank 0) and the last (final layers and the head, other ranks)
    groups = e.gather_buckets(w.gather_bucket)
    check_fetch_many(e, plan, w, T, None, [groups[0], groups[-1]], lambda i: ps.param[i],
                     state_ranks=[0], n=600)


def test_ragged_2000_full():
    """2000 ragged tensors, N_d = 7: shard offsets not multiples of 8 (element
    path), padding, shards crossing tensors, per-submodule fetch."""
    w = W.ragged()
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    T = 5
    e = run(w, T)
    check_sample(e, plan, w, sample_indices(plan, 0, plan.psi_pad, 100_000, 4), T)
    # persistent group (~5M elements) on a sample, ends included
    rng = np.random.default_rng(5)
    pidx = np.unique(np.concatenate([rng.integers(0, plan.psi_s, 50_000), [0, plan.psi_s - 1]]))
    p, m, v, h = sampled_persistent_oracle(w, plan, pidx, T)
    sel = torch.from_numpy(pidx).to(e.pmaster.device)
    for name, got, ref in (("pmaster", e.pmaster, p), ("pm", e.pm, m), ("pv", e.pv, v)):
        g = f32(got[sel])
        assert_f32_close(g, ref, what=name)
        assert np.array_equal(bits(g), bits(ref)), name
    assert np.array_equal(u16(e.pparam[sel]), h)
    # fetch: persistent members of the checked submodules come from the same sample set
    ps_param = np.zeros(plan.psi_s, np.uint16)
    ks = [0, 100, plan.n_submodules - 1]
    need = [np.arange(plan.offset[t], plan.offset[t] + plan.numel[t])
            for k in ks for t in plan.submodules[k] if plan.persistent[t]]
    if need:
        need = np.unique(np.concatenate(need))
        ps_param[need] = sampled_persistent_oracle(w, plan, need, T)[3]
    check_fetch(e, plan, w, T, None, ks, O.PersistState(None, None, None, ps_param))
    # the bench's bucketed gathers (several 512-piece launches per call)
    groups = e.gather_buckets(w.gather_bucket)
    check_fetch_many(e, plan, w, T, None, [groups[0]],
                     lambda i: sampled_persistent_oracle(w, plan, i, T)[3], n=200)


def test_llama_7b_full_emulation_max_size():
    """Maximum size: all 8 ranks of the Llama-7B list in one HBM (about 216
    GB: 108 GB of gradients, 81 GB of states, two 13.5 GB bf16 buffers),
    bucketed launches; flat offsets and all-gather offsets run past 2^32
    elements' bytes and 2^31 elements.  One step, sampled across every rank."""
    w = W.llama_7b(rank0_view=False)
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    assert plan.psi_pad > 2 ** 32
    e = run(w, 1, bucketed=True)
    idx = sample_indices(plan, 0, plan.psi_pad, 60_000, 6)
    assert idx.max() > 2 ** 32
    check_sample(e, plan, w, idx, 1)
    check_persistent(e, persistent_oracle(w, plan, 1))
