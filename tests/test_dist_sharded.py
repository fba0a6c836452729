"""One rank per process, on CPU: world sizes 2 and 3 under gloo run the
rank-per-process sharded step (all-to-all of the gradient slices, the local
update, all-gather of the bf16 shards) and every rank's state and `full`
buffer equal the oracle's one-process sharded step bit for bit.  There is no
GPU here, so each rank's local update is the oracle's own per-rank
arithmetic (reduce in rank order, AdamW, bf16 cast; the persistent group
DDP-style); what the test pins is the exchange and the gather around it:
which slice goes where, the padding, the persistent group and the gathered
layout."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _np_u16(t):
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)


def oracle_local_step(rk, t):
    """Rank rk.rank's update with the oracle's functions (CPU tensors)."""
    import oracle as O
    sc = O.adamw_scalars(rk.w.hparams, t, rk.nd)
    slices = [_np_u16(rk.slice_of(q)) for q in range(rk.nd)]
    g = O.reduce_sum(slices, sc["inv_nd"])
    p, m, v = O.adamw_update(g, rk.master.numpy().copy(), rk.m.numpy().copy(),
                             rk.v.numpy().copy(), sc)
    rk.master.copy_(torch.from_numpy(p))
    rk.m.copy_(torch.from_numpy(m))
    rk.v.copy_(torch.from_numpy(v))
    rk.sparam.copy_(_bf(O.cast_bf16(p)))
    if rk.psi_s:
        ps = O.PersistState(rk.pmaster.numpy().copy(), rk.pm.numpy().copy(),
                            rk.pv.numpy().copy(), _np_u16(rk.pparam))
        O.persistent_step(rk.oplan, rk.w.hparams, t, [_np_u16(rk.persist_of(q)) for q in range(rk.nd)],
                          ps, replicas=1)
        rk.pmaster.copy_(torch.from_numpy(ps.master))
        rk.pm.copy_(torch.from_numpy(ps.m))
        rk.pv.copy_(torch.from_numpy(ps.v))
        rk.pparam.copy_(_bf(ps.param))


def _worker(rank, world, port, wname, T, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle as O
    from tests._oracle_runs import host_grads, host_master, host_pgrads
    from zero_sharded_optimizer_shard_gb300 import workloads as W, zero3
    from zero_sharded_optimizer_shard_gb300.distributed import ShardedRank
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = {"ragged": lambda: W.ragged_small(world), "mini": lambda: W.mini_gpt(world)}[wname]()
    plan = zero3.Plan(w.numels, w.submodule_of, world, w.threshold, w.bucket)
    oplan = O.partition(w.numels, w.submodule_of, world, w.threshold, w.bucket)
    rk = ShardedRank(plan, zero3.hparams(**w.hparams), rank, device="cpu",
                     local_step=oracle_local_step)
    rk.w, rk.oplan = w, oplan
    S = rk.S
    mf, mp_ = host_master(w, oplan)
    rk.master.copy_(torch.from_numpy(mf[rank * S:(rank + 1) * S].copy()))
    rk.sparam.copy_(_bf(O.cast_bf16(rk.master.numpy())))
    rk.pmaster.copy_(torch.from_numpy(mp_))
    rk.pparam.copy_(_bf(O.cast_bf16(mp_)))
    rk.gather()  # the initial full buffer
    for t in range(1, T + 1):
        g = host_grads(w, oplan, t)[rank]
        pg = host_pgrads(w, oplan, t)[rank]
        rk.grad.copy_(_bf(np.concatenate([g, pg])))
        rk.step(t)
    out[rank] = {k: getattr(rk, k).numpy().copy() if getattr(rk, k).dtype == torch.float32
                 else _np_u16(getattr(rk, k))
                 for k in ("master", "m", "v", "sparam", "full", "pmaster", "pm", "pv", "pparam")}
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,wname", [(2, "ragged"), (3, "ragged"), (3, "mini")])
def test_rank_per_process_step_matches_oracle(world, wname, lib):
    from tests._oracle_runs import oracle_run
    from zero_sharded_optimizer_shard_gb300 import workloads as W
    T = 3
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), wname, T, out), nprocs=world,
                       join=True, start_method="spawn")
    w = {"ragged": lambda: W.ragged_small(world), "mini": lambda: W.mini_gpt(world)}[wname]()
    plan, st, full, ps = oracle_run(w, T)
    for r in range(world):
        got = out[r]
        for k in ("master", "m", "v"):
            assert np.array_equal(got[k].view(np.uint32), getattr(st, k)[r].view(np.uint32)), (r, k)
        assert np.array_equal(got["sparam"], st.sparam[r]), r
        assert np.array_equal(got["full"], full), r  # every rank holds the whole gathered buffer
        assert np.array_equal(got["pmaster"].view(np.uint32), ps.master.view(np.uint32)), r
        assert np.array_equal(got["pparam"], ps.param), r
