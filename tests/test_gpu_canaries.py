"""Guard-band canaries: every device buffer is surrounded by sentinel
elements (64 on each side) and every entry point that writes device memory
runs on ragged and aligned layouts; no band may change.  This checks the
kernels' bounds on the GPU without a memory sanitizer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from zero_sharded_optimizer_shard_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu
G = 64


def emu(w, **kw):
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    e = Emulation(w, guard=G, **kw)
    e.init_params()
    e.fill_grads(1)
    return e


def ok(e, what):
    torch.cuda.synchronize()
    bad = e.check_guards()
    assert not bad, f"{what}: guard bands written: {bad}"


@pytest.mark.parametrize("wname", ["ragged7", "mini8", "mini5"])
def test_every_writer_stays_in_bounds(wname, tmp_path):
    from zero_sharded_optimizer_shard_gb300 import zero3
    w = {"ragged7": lambda: W.ragged_small(7), "mini8": lambda: W.mini_gpt(8),
         "mini5": lambda: W.mini_gpt(5)}[wname]()
    w.bucket = 65_537  # odd bucket edges: element paths at every chunk start
    e = emu(w, bucketed=True)
    ok(e, "init / generator")
    P = e.ptrs
    for t in (1, 2):
        e.step(t)
    ok(e, "fused step + persistent (bucketed)")
    e.forward_backward_gathers()
    ok(e, "submodule gathers")
    total = sum(e.plan.submodule(k)[1] for k in range(e.plan.info.n_submodules))
    for div in (1, 4):  # every submodule in one call; buckets of a few
        e.forward_backward_gathers(bucket=max(1, total // div))
    ok(e, "bucketed submodule gathers (guarded arena)")
    nd, S = e.nd, e.S
    # unfused stages into guarded shard-gradient buffers, both dtypes
    for dt, torch_dt in ((zero3.F32, torch.float32), (zero3.BF16, torch.bfloat16)):
        sg = [e.alloc(S, torch_dt) for _ in range(nd)]
        for (lo, hi), Gr in zip(e.chunks, e.grads):
            zero3.zero3_reduce_scatter(e.plan, P(Gr), lo, lo, hi, P(sg), dt, e.sid)
        zero3.zero3_adamw_step(e.plan, e.hp, 3, P(sg), dt, P(e.master), P(e.m), P(e.v),
                               P(e.sparam), 0, e.psi_pad, e.sid)
        ok(e, f"reduce_scatter / adamw ({torch_dt})")
    zero3.zero3_allgather(e.plan, P(e.sparam), e.full.data_ptr(), 0, e.psi_pad, e.sid)
    zero3.zero3_cast_params(e.plan, P(e.master), P(e.sparam), e.full.data_ptr(), e.persist, 0,
                            e.psi_pad, e.sid)
    ok(e, "allgather / cast")
    # ZeRO-1/2 step into guarded full copies
    params = [e.alloc(e.psi_pad, torch.bfloat16) for _ in range(nd)]
    for (lo, hi), Gr in zip(e.chunks, e.grads):
        zero3.zero3_step_stage12(e.plan, e.hp, 4, P(Gr), lo, P(e.master), P(e.m), P(e.v),
                                 P(params), lo, hi, e.sid)
    ok(e, "stage 1/2 step")
    # qwZ needs block-aligned ranges: one launch over the whole flat range
    q = emu(w)
    nb = -(-S // 256)
    codes = [q.alloc(S, torch.int8) for _ in range(nd)]
    scales = [q.alloc(nb, torch.float32) for _ in range(nd)]
    for bits in (8, 4):
        cb = [q.alloc(-(-S * bits // 8), torch.int8) for _ in range(nd)]
        zero3.zero3_step_qwz(q.plan, q.hp, 1, P(q.grads[0]), 0, P(q.master), P(q.m), P(q.v),
                             P(q.sparam), P(cb), P(scales), q.persist, 0, q.psi_pad, q.sid,
                             bits=bits)
        zero3.zero3_quantize_shards(q.plan, P(q.sparam), P(cb), P(scales), 0, q.psi_pad, q.sid,
                                    bits=bits)
        zero3.zero3_allgather_qwz(q.plan, P(cb), P(scales), q.full.data_ptr(), 0, q.psi_pad,
                                  q.sid, bits=bits)
        ok(q, f"qwZ int{bits}")
    del q, codes, scales
    # checkpoint round trip writes the states back through host staging
    for r in range(nd):
        path = tmp_path / f"r{r}.ckpt"
        zero3.zero3_save_shard(e.plan, r, 5, e.master[r].data_ptr(), e.m[r].data_ptr(),
                               e.v[r].data_ptr(), path, e.sid)
        zero3.zero3_load_shard(e.plan, r, e.master[r].data_ptr(), e.m[r].data_ptr(),
                               e.v[r].data_ptr(), path, e.sid)
    ok(e, "checkpoint load")
    # prefetching coordinator into a guarded arena
    sizes = [e.plan.submodule(k)[1] for k in range(e.plan.info.n_submodules)]
    n_arena = (2 * max(sizes) + 7) // 8 * 8 + 8  # + 8: ranges of odd sizes leave gaps
    arena = e.alloc(n_arena, torch.bfloat16)
    compute, prefetch = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    co = zero3.Coordinator(e.plan, [], P(e.sparam), e.pparam.data_ptr(), arena.data_ptr(), n_arena,
                           max_live_parameters=n_arena, compute_stream=compute.cuda_stream,
                           prefetch_stream=prefetch.cuda_stream)
    order = list(range(len(sizes))) + list(reversed(range(len(sizes))))
    for step in range(2):
        for k in order:
            co.fetch(k)
            co.release(k)
        co.next_step()
    ok(e, "coordinator")
