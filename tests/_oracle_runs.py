"""Runs the CPU oracle on the seeded synthetic inputs of a workload, and
converts device buffers for comparison.  Test infrastructure."""
from __future__ import annotations

import numpy as np

import oracle as O
from zero_sharded_optimizer_shard_gb300 import synth
from zero_sharded_optimizer_shard_gb300.workloads import (STREAM_GRAD, STREAM_GRAD_PERSIST,
                                                          STREAM_MASTER, STREAM_MASTER_PERSIST)


def host_master_persist(w, plan):
    return synth.normal_f32(w.seed, STREAM_MASTER_PERSIST, 0, 0, np.arange(plan.psi_s),
                            w.master_sigma)


def host_master(w, plan):
    mf = np.zeros(plan.psi_pad, np.float32)
    mf[:plan.psi_p] = synth.normal_f32(w.seed, STREAM_MASTER, 0, 0, np.arange(plan.psi_p),
                                       w.master_sigma)
    return mf, host_master_persist(w, plan)


def host_grads(w, plan, t, idx=None):
    """Every rank's bf16 local gradient at step t (full flat buffer with zero
    padding, or only at flat indices idx)."""
    out = []
    for q in range(plan.n_ranks):
        if idx is None:
            g = np.zeros(plan.psi_pad, np.uint16)
            g[:plan.psi_p] = synth.normal_bf16(w.seed, STREAM_GRAD, t, q, np.arange(plan.psi_p),
                                               w.grad_sigma, w.outlier_p, w.outlier_sigma)
        else:
            g = synth.normal_bf16(w.seed, STREAM_GRAD, t, q, idx, w.grad_sigma, w.outlier_p,
                                  w.outlier_sigma)
            g[idx >= plan.psi_p] = 0
        out.append(g)
    return out


def host_pgrads(w, plan, t):
    return [synth.normal_bf16(w.seed, STREAM_GRAD_PERSIST, t, q, np.arange(plan.psi_s),
                              w.grad_sigma, w.outlier_p, w.outlier_sigma)
            for q in range(plan.n_ranks)]


def oracle_run(w, T, grad_step=None):
    """Whole-workload oracle: T sharded steps plus the persistent group.
    grad_step fixes the generator step of the gradients (None: step t)."""
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    mf, mp = host_master(w, plan)
    st, full, ps = O.init_state(plan, mf, mp)
    for t in range(1, T + 1):
        gs = t if grad_step is None else grad_step
        O.sharded_step(plan, w.hparams, t, host_grads(w, plan, gs), st, full)
        O.persistent_step(plan, w.hparams, t, host_pgrads(w, plan, gs), ps)
    return plan, st, full, ps


def sampled_oracle(w, plan, idx, T, grad_step=None):
    """Oracle for a sample of flat indices only (elementwise independence):
    returns master, m, v, bf16 param at idx after T steps."""
    idx = np.asarray(idx, np.int64)
    p = synth.normal_f32(w.seed, STREAM_MASTER, 0, 0, idx, w.master_sigma)
    p[idx >= plan.psi_p] = 0
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    for t in range(1, T + 1):
        gs = t if grad_step is None else grad_step
        sc = O.adamw_scalars(w.hparams, t, plan.n_ranks)
        g = O.reduce_sum(host_grads(w, plan, gs, idx), sc["inv_nd"])
        p, m, v = O.adamw_update(g, p, m, v, sc)
    return p, m, v, O.cast_bf16(p)


def sampled_persistent_oracle(w, plan, pidx, T, grad_step=None):
    """Persistent-group oracle at persistent indices pidx only."""
    pidx = np.asarray(pidx, np.int64)
    p = synth.normal_f32(w.seed, STREAM_MASTER_PERSIST, 0, 0, pidx, w.master_sigma)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    for t in range(1, T + 1):
        gs = t if grad_step is None else grad_step
        sc = O.adamw_scalars(w.hparams, t, plan.n_ranks)
        g = O.reduce_sum([synth.normal_bf16(w.seed, STREAM_GRAD_PERSIST, gs, q, pidx, w.grad_sigma,
                                            w.outlier_p, w.outlier_sigma)
                          for q in range(plan.n_ranks)], sc["inv_nd"])
        p, m, v = O.adamw_update(g, p, m, v, sc)
    return p, m, v, O.cast_bf16(p)


def u16(t):
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t):
    return t.detach().cpu().numpy()


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def assert_f32_close(got, ref, rel=2e-6, what=""):
    """|got - ref| <= rel * |ref|, with ref == 0 requiring got == 0; NaN
    positions must match."""
    got = np.asarray(got, np.float32)
    ref = np.asarray(ref, np.float32)
    assert got.shape == ref.shape, what
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ"
    ok = ~nan_r
    err = np.abs(got[ok].astype(np.float64) - ref[ok].astype(np.float64))
    bound = rel * np.abs(ref[ok].astype(np.float64))
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond {rel} relative, first at " \
                          f"{np.flatnonzero(ok)[np.argmax(bad)]}"


def assert_bf16_close(got, ref, ulps=1, what=""):
    """bf16 patterns within `ulps` units in the last place (same sign);
    NaN positions must match."""
    got = np.asarray(got, np.uint16)
    ref = np.asarray(ref, np.uint16)
    gf, rf = O.bf16_to_f32(got), O.bf16_to_f32(ref)
    assert np.array_equal(np.isnan(gf), np.isnan(rf)), f"{what}: NaN positions differ"
    ok = ~np.isnan(rf)
    # map sign-magnitude patterns onto a monotone integer line
    def line(u):
        u = u.astype(np.int64)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    d = np.abs(line(got[ok]) - line(ref[ok]))
    assert d.max(initial=0) <= ulps, f"{what}: max {d.max()} bf16 ulps"
