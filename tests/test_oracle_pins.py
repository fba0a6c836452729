"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test compares the oracle with something other than itself: numbers
printed on the pages (tests/golden), closed forms evaluated in float64, a
library routine (torch.optim.AdamW, torch's bf16 cast) and brute force.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle as O
from zero_sharded_optimizer_shard_gb300 import synth, workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HP = dict(W.ADAMW)


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16(x):
    return O.bf16_rne(np.asarray(x, np.float32))


def ulp32(x):
    x = np.abs(np.asarray(x, np.float64)).astype(np.float32)
    return (np.nextafter(x, np.float32(np.inf)) - x).astype(np.float64)


# ---------------------------------------------------------------- pages' worked examples
def test_reduce_scatter_worked_example():
    g = golden("reduce_scatter_example.json")
    plan = O.partition([2], None, 2, threshold=0)
    grads = [bf16(x) for x in g["local_grads"]]
    inv = O.adamw_scalars(HP, 1, 2)["inv_nd"]
    rs = O.reduce_scatter(plan, grads, inv)
    assert [list(map(float, s)) for s in rs] == [list(map(float, x)) for x in g["reduce_scatter"]]
    ar = O.reduce_sum(grads, inv)
    assert list(map(float, ar)) == list(map(float, g["allreduce_mean"]))


def test_two_parameter_example_allgather():
    g = golden("two_param_example.json")
    plan = O.partition([2], None, 2, threshold=0)
    shards = [bf16(s) for s in g["shard_updates"]]
    full = O.allgather(plan, shards)
    assert list(map(float, O.bf16_to_f32(full))) == [float(x) for x in g["after_gather"]]
    # before the gather each rank's local full copy holds only its own update
    before = bf16(g["before"])
    for r in range(2):
        view = before.copy()
        view[r * plan.shard_len:(r + 1) * plan.shard_len] = shards[r]
        assert list(map(float, O.bf16_to_f32(view))) == [float(x) for x in g["local_views_before_gather"][r]]


def test_eight_weights_on_four_gpus():
    g = golden("eight_weights_four_gpus.json")
    plan = O.partition([g["numel"]], None, g["n_ranks"], threshold=0)
    assert plan.shard_len == 2 and plan.psi_pad == 8
    owned = [[] for _ in range(g["n_ranks"])]
    for (r, so, to, ln) in plan.segments[0]:
        owned[r].extend(range(to, to + ln))
    assert owned == g["owned"]
    # gathering the layer returns w0..w7 in order
    w = np.arange(8, dtype=np.float32)
    sparam = [bf16(w[2 * r:2 * r + 2]) for r in range(4)]
    got = O.fetch_submodule(plan, 0, sparam, np.zeros(0, np.uint16))
    assert list(O.bf16_to_f32(got)) == list(w)


# ---------------------------------------------------------------- accounting
def test_memory_accounting_numbers():
    g = golden("accounting.json")
    for c in g["cases"]:
        b = O.memory_bytes(c["stage"], c["psi"], c["n_d"], g["bytes_per_param_K"])
        if "gb" in c:
            assert b == pytest.approx(c["gb"] * 1e9, rel=1e-12), c
        else:
            assert abs(b / 1e9 - c["gb_approx"]) <= c["abs_tol_gb"], c
    for c in g["fractions_nd64"]:
        frac = O.memory_bytes(c["stage"], 1.0, 64) / O.memory_bytes(0, 1.0, 64)
        assert abs(frac - c["approx"]) <= c["abs_tol"], c
    # exact closed forms of the same fractions
    assert O.memory_bytes(1, 1.0, 64) / 16 == 0.26171875
    assert O.memory_bytes(2, 1.0, 64) / 16 == 0.138671875
    assert O.memory_bytes(3, 1.0, 64) / 16 == 0.015625


def test_communication_accounting_numbers():
    g = golden("accounting.json")
    ring = g["ring_7b_4gpu_gb"]
    assert O.ring_send_bytes(2, 7e9, 4) == pytest.approx(ring["stage2"] * 1e9, rel=1e-12)
    assert O.ring_send_bytes(0, 7e9, 4) == pytest.approx(ring["ddp"] * 1e9, rel=1e-12)
    assert O.ring_send_bytes(3, 7e9, 4) == pytest.approx(ring["stage3"] * 1e9, rel=1e-12)
    assert O.comm_elems(3, 1.0) / O.comm_elems(0, 1.0) == g["comm_ratio_stage3_vs_dp"]


# ---------------------------------------------------------------- bf16 cast
def test_bf16_rne_matches_torch_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(0.02),
        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38,
                  1e-40, -1e-40, 1.17549435e-38, 65504.0], np.float32),
        # exact ties between two bf16 values: lower half 0x8000, both parities
        np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F80FFFF, 0x3F807FFF, 0x7F7FFFFF],
                 np.uint32).view(np.float32),
    ])
    ours = O.bf16_rne(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # ties to even: 1 + 2^-8 rounds down to 1, 1 + 3*2^-8 rounds up
    assert O.bf16_rne(np.array([0x3F808000], np.uint32).view(np.float32))[0] == 0x3F80
    assert O.bf16_rne(np.array([0x3F818000], np.uint32).view(np.float32))[0] == 0x3F82


def test_bf16_nan_stays_nan():
    x = np.array([np.nan, -np.nan, np.array(0x7F800001, np.uint32).view(np.float32)], np.float32)
    r = O.bf16_to_f32(O.bf16_rne(x))
    assert np.isnan(r).all()


# ---------------------------------------------------------------- AdamW closed forms
def _scalar_run(gs, p0, hp=HP, n_ranks=1):
    """Run the oracle's elementwise update on one element per column."""
    p = np.asarray(p0, np.float32).copy()
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    for t, g in enumerate(gs, start=1):
        sc = O.adamw_scalars(hp, t, n_ranks)
        p, m, v = O.adamw_update(np.asarray(g, np.float32), p, m, v, sc)
    return p, m, v


def test_adamw_first_step_closed_form():
    """t=1, m0=v0=0: m_hat = g and v_hat = g^2 exactly, so
    p1 = p0 (1 - lr wd) - lr g / (|g| + eps) (float64)."""
    rng = np.random.default_rng(1)
    p0 = (rng.standard_normal(4096) * 0.02).astype(np.float32)
    g = np.concatenate([rng.standard_normal(2048) * 1e-3,
                        rng.standard_normal(2048) * 1e-8]).astype(np.float32)
    p1, m1, v1 = _scalar_run([g], p0)
    lr, wd, eps = HP["lr"], HP["weight_decay"], HP["eps"]
    gd = g.astype(np.float64)
    exact = p0.astype(np.float64) * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
    # rounding-error bound: p*decay (incl. the rounded decay constant) costs
    # at most one ulp of p0, the final subtraction half an ulp of p1, and the
    # update term a few binary32 ulps relative to lr
    bound = ulp32(p0) + ulp32(exact) + 1e-6 * lr
    assert np.all(np.abs(p1 - exact) <= bound)
    assert np.allclose(m1, (1 - HP["beta1"]) * gd, rtol=2e-7, atol=0)
    assert np.allclose(v1, (1 - HP["beta2"]) * gd * gd, rtol=4e-7, atol=0)


def test_adamw_ten_steps_explicit_sums():
    """Closed form of T steps with varying gradients, evaluated in float64:
    m_T = (1-b1) sum_k b1^(T-k) g_k, v_T = (1-b2) sum_k b2^(T-k) g_k^2,
    p_T = decay^T p0 - lr sum_t decay^(T-t) m_hat_t / (sqrt(v_hat_t) + eps).
    Catches dropped bias corrections, swapped betas, eps placement, sign."""
    rng = np.random.default_rng(2)
    T, n = 10, 4096
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    gs = [(rng.standard_normal(n) * np.where(np.arange(n) < n // 2, 1e-3, 3e-8)).astype(np.float32)
          for _ in range(T)]
    pT, mT, vT = _scalar_run(gs, p0)
    b1, b2, lr, wd, eps = HP["beta1"], HP["beta2"], HP["lr"], HP["weight_decay"], HP["eps"]
    G = np.stack([g.astype(np.float64) for g in gs])
    decay = 1 - lr * wd
    p = p0.astype(np.float64) * decay ** T
    for t in range(1, T + 1):
        m_t = (1 - b1) * sum(b1 ** (t - k) * G[k - 1] for k in range(1, t + 1))
        v_t = (1 - b2) * sum(b2 ** (t - k) * G[k - 1] ** 2 for k in range(1, t + 1))
        u = (m_t / (1 - b1 ** t)) / (np.sqrt(v_t / (1 - b2 ** t)) + eps)
        p -= lr * decay ** (T - t) * u
    m_exact = (1 - b1) * sum(b1 ** (T - k) * G[k - 1] for k in range(1, T + 1))
    v_exact = (1 - b2) * sum(b2 ** (T - k) * G[k - 1] ** 2 for k in range(1, T + 1))
    # error bound accumulated over T steps (see the first-step test)
    bound = 2 * T * ulp32(np.maximum(np.abs(p0), np.abs(p))) + 1e-6 * lr * T
    assert np.all(np.abs(pT - p) <= bound)
    scale_m = np.max(np.abs(G), axis=0)
    assert np.all(np.abs(mT - m_exact) <= 1e-6 * scale_m)
    assert np.allclose(vT, v_exact, rtol=4e-6, atol=0)


def test_single_rank_reduces_to_torch_adamw():
    """N_d = 1, threshold 0: the sharded step is plain AdamW on one flat
    tensor; compare with torch.optim.AdamW (fp32, for-loop implementation)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    n, T = 10000, 10
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    plan = O.partition([n], None, 1, threshold=0)
    st, full, _ = O.init_state(plan, p0, np.zeros(0, np.float32))
    w = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([w], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"], foreach=False, fused=False)
    for t in range(1, T + 1):
        g16 = bf16((rng.standard_normal(n) * 1e-3).astype(np.float32))
        O.sharded_step(plan, HP, t, [g16], st, full)
        w.grad = torch.from_numpy(O.bf16_to_f32(g16).copy())
        opt.step()
    ref_p = w.detach().numpy()
    s = opt.state[w]
    # different op order (lerp for m, divide by sqrt(bc2)): the two may differ
    # by a few roundings per step, in ulps of max(|p|, lr)
    scale = ulp32(np.maximum(np.maximum(np.abs(p0), np.abs(ref_p)), HP["lr"]))
    assert np.all(np.abs(st.master[0] - ref_p) <= 2 * T * scale)
    m_ref, v_ref = s["exp_avg"].numpy(), s["exp_avg_sq"].numpy()
    assert np.all(np.abs(st.m[0] - m_ref) <= 1e-6 * np.abs(m_ref) + 1e-6 * np.abs(m_ref).max())
    assert np.allclose(st.v[0], v_ref, rtol=1e-6, atol=0)


# ---------------------------------------------------------------- invariants
def _random_problem(numels, nd, seed, threshold=100):
    plan = O.partition(numels, None, nd, threshold=threshold)
    mf = np.zeros(plan.psi_pad, np.float32)
    idx = np.arange(plan.psi_p)
    mf[:plan.psi_p] = synth.normal_f32(seed, 1, 0, 0, idx, 0.02)
    mp = synth.normal_f32(seed, 2, 0, 0, np.arange(plan.psi_s), 0.02)
    return plan, mf, mp


def _grads(plan, seed, t, nd):
    G = []
    for q in range(nd):
        g = np.zeros(plan.psi_pad, np.uint16)
        g[:plan.psi_p] = synth.normal_bf16(seed, 3, t, q, np.arange(plan.psi_p), 1e-3, 0.01, 0.1)
        G.append(g)
    return G


@pytest.mark.parametrize("nd", [1, 2, 3, 4, 7, 8])
def test_sharded_equals_ddp_bitwise(nd):
    """Sharded update + all-gather == full redundant DDP update, bit for bit
    ("ddp-to-zero-memory-sharding", section "ZeRO-1": AdamW updates of
    different parameters are independent; ZeRO concept page, comparison
    table: no precision impact for ZeRO-3)."""
    numels = [1000, 37, 5, 2300, 999, 64]
    plan, mf, _ = _random_problem(numels, nd, seed=11)
    st, full, _ = O.init_state(plan, mf, np.zeros(0, np.float32))
    ddp = O.ddp_init(plan, mf)
    for t in range(1, 6):
        G = _grads(plan, 11, t, nd)
        O.sharded_step(plan, HP, t, G, st, full)
        O.ddp_step(plan, HP, t, G, ddp)
        assert np.array_equal(np.concatenate(st.master).view(np.uint32), ddp.master[0].view(np.uint32))
        assert np.array_equal(np.concatenate(st.m).view(np.uint32), ddp.m[0].view(np.uint32))
        assert np.array_equal(np.concatenate(st.v).view(np.uint32), ddp.v[0].view(np.uint32))
        assert np.array_equal(full, ddp.param[0])


@pytest.mark.parametrize("nd", [2, 3, 8])
def test_stage12_replicas_equal_ddp(nd):
    """ZeRO-1/2: after every step each rank's full parameter copy equals the
    DDP replicas' parameters (the all-gather restores consistency:
    "ddp-to-zero-memory-sharding", section "ZeRO-1")."""
    numels = [1000, 37, 5, 2300, 999, 64]
    plan, mf, _ = _random_problem(numels, nd, seed=12, threshold=0)
    st, full, _ = O.init_state(plan, mf, np.zeros(0, np.float32))
    params = [full.copy() for _ in range(nd)]
    ddp = O.ddp_init(plan, mf)
    for t in range(1, 4):
        G = _grads(plan, 12, t, nd)
        O.replicated_step(plan, HP, t, G, st, params)
        O.ddp_step(plan, HP, t, G, ddp)
        for q in range(nd):
            assert np.array_equal(params[q], ddp.param[q])
        assert np.array_equal(np.concatenate(st.master).view(np.uint32), ddp.master[0].view(np.uint32))


def test_padding_stays_zero():
    plan, mf, _ = _random_problem([1001, 13], 4, seed=5, threshold=0)
    assert plan.psi_pad - plan.psi_p == 2
    st, full, _ = O.init_state(plan, mf, np.zeros(0, np.float32))
    for t in range(1, 4):
        O.sharded_step(plan, HP, t, _grads(plan, 5, t, 4), st, full)
    flat = np.concatenate(st.master)
    assert not flat[plan.psi_p:].view(np.uint32).any()
    assert not full[plan.psi_p:].any()


@pytest.mark.parametrize("bucket", [1, 7, 64, 333, 10**9])
def test_bucket_invariance(bucket):
    numels = [700, 3, 1200, 55]
    plan, mf, _ = _random_problem(numels, 3, seed=9)
    plan_b = O.partition(numels, None, 3, threshold=100, bucket=bucket)
    st1, full1, _ = O.init_state(plan, mf, np.zeros(0, np.float32))
    st2, full2, _ = O.init_state(plan_b, mf, np.zeros(0, np.float32))
    for t in range(1, 4):
        G = _grads(plan, 9, t, 3)
        O.sharded_step(plan, HP, t, G, st1, full1)
        for lo, hi in plan_b.buckets:
            O.sharded_step(plan_b, HP, t, G, st2, full2, lo, hi)
    assert np.array_equal(np.concatenate(st1.master), np.concatenate(st2.master))
    assert np.array_equal(full1, full2)


def test_threshold_is_strict():
    plan = O.partition([99_999, 100_000, 100_001], None, 2, threshold=100_000)
    assert plan.persistent == [True, False, False]


def test_persistent_replicas_agree_and_match_ddp():
    rng = np.random.default_rng(4)
    n, nd = 300, 5
    plan = O.partition([n], None, nd, threshold=10**6)
    assert plan.persistent == [True] and plan.psi_s == n and plan.psi_pad == 0
    mp = (rng.standard_normal(n) * 0.02).astype(np.float32)
    ps = O.PersistState(mp.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), O.bf16_rne(mp))
    plan_d = O.partition([n], None, nd, threshold=0)
    ddp = O.ddp_init(plan_d, np.concatenate([mp, np.zeros(plan_d.psi_pad - n, np.float32)]))
    for t in range(1, 4):
        pg = [O.bf16_rne((rng.standard_normal(n) * 1e-3).astype(np.float32)) for _ in range(nd)]
        O.persistent_step(plan, HP, t, pg, ps)
        O.ddp_step(plan_d, HP, t, [np.concatenate([g, np.zeros(plan_d.psi_pad - n, np.uint16)]) for g in pg], ddp)
    assert np.array_equal(ps.master, ddp.master[0][:n])
    assert np.array_equal(ps.param, ddp.param[0][:n])


# ---------------------------------------------------------------- brute force of the shard map
def _brute_partition(numels, nd, thr):
    """Build the flat buffer as an explicit list of (tensor, element) labels,
    pad it with None, and cut it into nd equal lists."""
    flat = [(t, e) for t, n in enumerate(numels) if n >= thr for e in range(n)]
    while len(flat) % nd:
        flat.append(None)
    S = len(flat) // nd
    return [flat[r * S:(r + 1) * S] for r in range(nd)], S


@pytest.mark.parametrize("nd", list(range(1, 10)))
def test_partition_brute_force(nd):
    rng = np.random.default_rng(100 + nd)
    for trial in range(60):
        n_t = int(rng.integers(0, 7))
        numels = [int(x) for x in rng.integers(0, 13, n_t)]
        thr = int(rng.integers(0, 8))
        bucket = int(rng.integers(1, 20))
        plan = O.partition(numels, None, nd, threshold=thr, bucket=bucket)
        shards, S = _brute_partition(numels, nd, thr)
        assert plan.shard_len == S
        rebuilt = [[None] * S for _ in range(nd)]
        for t, segs in enumerate(plan.segments):
            covered = 0
            for (r, so, to, ln) in segs:
                assert 0 < ln and 0 <= so and so + ln <= S
                for e in range(ln):
                    rebuilt[r][so + e] = (t, to + e)
                covered += ln
            assert covered == (numels[t] if numels[t] >= thr else 0)
        assert rebuilt == shards
        # persistent offsets: running sum in list order
        po = 0
        for t, n in enumerate(numels):
            if n < thr:
                assert plan.persistent[t] and plan.offset[t] == po
                po += n
        assert plan.psi_s == po
        # buckets tile [0, psi_pad) exactly
        edges = [x for b in plan.buckets for x in b]
        assert (not plan.buckets and plan.psi_pad == 0) or (edges[0] == 0 and edges[-1] == plan.psi_pad)
        for (a, b), (c, d) in zip(plan.buckets, plan.buckets[1:]):
            assert b == c and b - a == bucket
        # fetch reproduces every tensor element from the owning shard
        vals = [np.arange(1, n + 1, dtype=np.uint16) * np.uint16(t + 1) for t, n in enumerate(numels)]
        sparam = [np.array([0 if lab is None else vals[lab[0]][lab[1]] for lab in shards[r]], np.uint16)
                  for r in range(nd)]
        pp = np.concatenate([vals[t] for t in range(n_t) if numels[t] < thr] + [np.zeros(0, np.uint16)])
        for t in range(n_t):
            got = O.fetch_submodule(plan, t, sparam, pp)
            assert np.array_equal(got, vals[t])
        # consolidated 16-bit weights: every tensor complete, in list order
        whole = O.gather_16bit_weights(plan, sparam, pp)
        assert len(whole) == n_t and all(np.array_equal(a, b) for a, b in zip(whole, vals))
        # the fp32 merge uses the same mapping on float shards
        fvals = [v.astype(np.float32) * np.float32(0.5) for v in vals]
        fsh = [np.array([0 if lab is None else fvals[lab[0]][lab[1]] for lab in shards[r]], np.float32)
               for r in range(nd)]
        fpp = np.concatenate([fvals[t] for t in range(n_t) if numels[t] < thr] + [np.zeros(0, np.float32)])
        merged = O.merge_fp32_weights(plan, fsh, fpp)
        assert all(np.array_equal(a, b) for a, b in zip(merged, fvals))


def test_workload_sizes():
    """Sizes of the model-shaped lists (parameter counts of the named
    architectures) and the derived shard lengths."""
    cases = {
        "toy": (W.toy_mlp(), 1_068_810, 1_064_960, 3_850, 532_480),
        "gpt2": (W.gpt2_small(), 124_439_808, 124_318_464, 121_344, 31_079_616),
        "1.3b": (W.decoder_1p3b(), 1_315_723_264, 1_315_080_192, 643_072, 164_385_024),
        "7b": (W.llama_7b(), 6_738_415_616, 6_738_149_376, 266_240, 842_268_672),
    }
    for name, (w, psi, psi_p, psi_s, S) in cases.items():
        plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
        assert (w.psi, plan.psi_p, plan.psi_s, plan.shard_len) == (psi, psi_p, psi_s, S), name


def test_ragged_list_recipe():
    w = W.ragged()
    assert len(w.numels) == 2000
    assert all(n % 7 for n in w.numels)
    frac_small = sum(n < 100_000 for n in w.numels) / 2000
    assert 0.25 < frac_small < 0.35
    plan = O.partition(w.numels, w.submodule_of, 7)
    assert plan.psi_pad - plan.psi_p in range(0, 7)
    assert max(w.submodule_of) + 1 == len(set(w.submodule_of))
    runs = np.bincount(w.submodule_of)
    assert runs.min() >= 1 and runs.max() <= 8


def test_ragged_list_one_rank_terminates():
    # every size is divisible by one rank: nothing is redrawn
    w = W.ragged_small(1)
    assert len(w.numels) == 300 and w.n_ranks == 1


def test_state_machine():
    sm = O.SubmoduleStates(2)
    assert sm.fetch(0) is True and sm.status[0] == O.INFLIGHT
    sm.complete(0)
    assert sm.status[0] == O.AVAILABLE
    assert sm.fetch(0) is False and sm.refs[0] == 2
    sm.release(0)
    assert sm.status[0] == O.AVAILABLE
    sm.release(0)
    assert sm.status[0] == O.NOT_AVAILABLE
    with pytest.raises(RuntimeError):
        sm.release(1)


# ---------------------------------------------------------------- qwZ quantized all-gather
def test_qwz_hand_example():
    g = golden("qwz_block_example.json")
    codes, scales = O.qwz_quantize(bf16(g["x"]), block=g["block"])
    assert list(codes) == g["codes"]
    assert scales[0] == np.float32(g["absmax"]) / np.float32(127)
    deq = O.bf16_to_f32(O.qwz_dequantize(codes, scales, block=g["block"]))
    assert list(map(float, deq)) == g["dequant"]


def test_qwz_error_bound_and_extremes():
    """Per element |dequant - x| <= scale/2 (rounding of the code) plus the
    binary32 product and the bf16 rounding of the result; the block's absmax
    element maps to +-127; an all-zero block gives zero codes and scale."""
    rng = np.random.default_rng(21)
    x16 = bf16((rng.standard_normal(10_000) * 0.02).astype(np.float32))
    x16[256:512] = 0
    codes, scales = O.qwz_quantize(x16)
    x = O.bf16_to_f32(x16).astype(np.float64)
    y = O.bf16_to_f32(O.qwz_dequantize(codes, scales)).astype(np.float64)
    s = np.repeat(scales.astype(np.float64), 256)[:x.size]
    bound = s / 2 * (1 + 1e-6) + np.abs(x) * 2.0 ** -8 + 1e-45
    assert np.all(np.abs(y - x) <= bound)
    assert np.all(np.abs(codes.astype(int)) <= 127)
    for b in range(scales.size):
        blk = np.abs(x[b * 256:(b + 1) * 256])
        if blk.max() > 0:
            assert np.abs(codes[b * 256:(b + 1) * 256]).max() == 127
        else:
            assert scales[b] == 0 and not codes[b * 256:(b + 1) * 256].any()
    assert scales.size == -(-10_000 // 256)  # last block partial


def test_qwz_allgather_layout():
    plan = O.partition([1000, 700], None, 3, threshold=0)
    rng = np.random.default_rng(3)
    shards = [bf16(rng.standard_normal(plan.shard_len).astype(np.float32)) for _ in range(3)]
    q = [O.qwz_quantize(s) for s in shards]
    full = O.qwz_allgather(plan, [c for c, _ in q], [s for _, s in q])
    S = plan.shard_len
    for r in range(3):
        assert np.array_equal(full[r * S:(r + 1) * S], O.qwz_dequantize(*q[r]))


def test_plan_memory_reduces_to_closed_form():
    """No persistent tensors and no padding: the plan's per-rank bytes are
    the closed forms; the 7B / 4-GPU plan gives the pages' 28 GB at stage 3.
    Padding and persistent tensors add exactly their own bytes."""
    plan = O.partition([7_000_000_000], None, 4, threshold=0)
    assert O.plan_memory_bytes(plan, 3) == 28e9
    assert O.plan_memory_bytes(plan, 2) == 38.5e9
    assert O.plan_memory_bytes(plan, 1) == 49e9
    assert O.plan_memory_bytes(plan, 0) == 112e9
    plan = O.partition([1001, 50], None, 4, threshold=100)
    assert plan.psi_pad == 1004 and plan.psi_s == 50
    assert O.plan_memory_bytes(plan, 3) == 16 * 1004 / 4 + 16 * 50


def test_qwz_int4_hand_example():
    g = golden("qwz_int4_block_example.json")
    codes, scales = O.qwz_quantize(bf16(g["x"]), block=g["block"], bits=4)
    assert list(codes) == g["codes"]
    assert list(O.qwz_pack(codes, bits=4)) == g["packed"]
    assert list(O.qwz_unpack(O.qwz_pack(codes, bits=4), len(codes), bits=4)) == g["codes"]
    deq = O.bf16_to_f32(O.qwz_dequantize(codes, scales, block=g["block"]))
    assert list(map(float, deq)) == g["dequant"]


def test_qwz_int4_error_bound():
    rng = np.random.default_rng(22)
    x16 = bf16((rng.standard_normal(5_000) * 0.02).astype(np.float32))
    codes, scales = O.qwz_quantize(x16, bits=4)
    assert np.abs(codes.astype(int)).max() <= 7
    x = O.bf16_to_f32(x16).astype(np.float64)
    y = O.bf16_to_f32(O.qwz_dequantize(codes, scales)).astype(np.float64)
    s = np.repeat(scales.astype(np.float64), 256)[:x.size]
    assert np.all(np.abs(y - x) <= s / 2 * (1 + 1e-6) + np.abs(x) * 2.0 ** -8 + 1e-45)
    # pack/unpack round trip for both widths, odd and even lengths
    for bits in (8, 4):
        for n in (5_000, 4_999):
            c = codes[:n]
            assert np.array_equal(O.qwz_unpack(O.qwz_pack(c, bits), n, bits), c)
