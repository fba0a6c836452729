"""The rank-per-process step's CUDA part on one GPU: each rank's local update
(zero3_step over its own flat range, gradients read from the received
slices, the persistent group from the gathered persistent gradients) against
the oracle.  The ranks' collectives are emulated by device copies, one phase
for all ranks before the next, so no kernel waits on another; and a real
NCCL process group of world size 1 runs the whole step with its
collectives."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from tests._oracle_runs import (bits, f32, host_grads, host_master, host_pgrads,  # noqa: E402
                                oracle_run, u16)
from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)


def _init(rk, w, oplan):
    mf, mp = host_master(w, oplan)
    S, r = rk.S, rk.rank
    rk.master.copy_(torch.from_numpy(mf[r * S:(r + 1) * S].copy()))
    rk.pmaster.copy_(torch.from_numpy(mp))
    rk.cast_params()


def _compare(ranks, plan, st, full, ps):
    for rk in ranks:
        r = rk.rank
        for k in ("master", "m", "v"):
            assert np.array_equal(bits(f32(getattr(rk, k))), bits(getattr(st, k)[r])), (r, k)
        assert np.array_equal(u16(rk.sparam), st.sparam[r]), r
        assert np.array_equal(u16(rk.full), full), r
        assert np.array_equal(bits(f32(rk.pmaster)), bits(ps.master)), r
        assert np.array_equal(u16(rk.pparam), ps.param), r


@pytest.mark.parametrize("nd,wname", [(2, "ragged"), (3, "mini"), (7, "ragged")])
def test_every_rank_local_step_matches_oracle(lib, nd, wname):
    import oracle as O
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.distributed import ShardedRank
    w = {"ragged": lambda: W.ragged_small(nd), "mini": lambda: W.mini_gpt(nd)}[wname]()
    T = 3
    plan = zero3.Plan(w.numels, w.submodule_of, nd, w.threshold, w.bucket)
    oplan = O.partition(w.numels, w.submodule_of, nd, w.threshold, w.bucket)
    hp = zero3.hparams(**w.hparams)
    ranks = [ShardedRank(plan, hp, r, device="cuda") for r in range(nd)]
    S, pad = ranks[0].S, ranks[0].psi_pad

    def gather():  # every rank's shard into every rank's full buffer
        cat = torch.cat([rk.sparam for rk in ranks])
        for rk in ranks:
            rk.full.copy_(cat)

    for rk in ranks:
        _init(rk, w, oplan)
    gather()
    for t in range(1, T + 1):
        G = [_bf(np.concatenate([g, pg])).cuda() for g, pg in
             zip(host_grads(w, oplan, t), host_pgrads(w, oplan, t))]
        for rk in ranks:  # the all-to-all of the gradient slices and persistent gradients
            for q in range(nd):
                rk.slice_of(q).copy_(G[q][rk.rank * S:(rk.rank + 1) * S])
                rk.persist_of(q).copy_(G[q][pad:])
        for rk in ranks:
            rk.fused_step(t)
        gather()
    torch.cuda.synchronize()
    plan_o, st, full, ps = oracle_run(w, T)
    _compare(ranks, plan_o, st, full, ps)


def test_world_size_one_with_nccl(lib):
    """The whole step through torch.distributed (NCCL, one rank)."""
    import oracle as O
    import torch.distributed as dist
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.distributed import ShardedRank
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        w = W.mini_gpt(1)
        plan = zero3.Plan(w.numels, w.submodule_of, 1, w.threshold, w.bucket)
        oplan = O.partition(w.numels, w.submodule_of, 1, w.threshold, w.bucket)
        rk = ShardedRank(plan, zero3.hparams(**w.hparams), 0, device="cuda")
        _init(rk, w, oplan)
        rk.gather()
        for t in range(1, 4):
            rk.grad.copy_(_bf(np.concatenate([host_grads(w, oplan, t)[0],
                                              host_pgrads(w, oplan, t)[0]])).cuda())
            rk.step(t)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    plan_o, st, full, ps = oracle_run(w, 3)
    _compare([rk], plan_o, st, full, ps)
