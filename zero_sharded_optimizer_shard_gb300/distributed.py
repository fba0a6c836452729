"""One data-parallel rank per process: the sharded step across real ranks.

The one-GPU emulation keeps every rank's buffers in one HBM; here each
process (one GPU each, or a CPU process in tests) owns one rank r of N_d and
the ranks exchange data through torch.distributed collectives (NCCL on GPUs,
gloo on CPU).  The pages' per-step flow ("ddp-to-zero-memory-sharding",
section "ZeRO-2：梯度为什么也可以分片"; ZERO tutorial, cnhsyj.com, section
2.2; "ZeRO-1/2/3" concept page, "ZeRO Stage 3 的 AllGather 與釋放機制"):

  1. reduce-scatter of the bf16 local gradients.  Its communication is one
     all-to-all: rank r receives slice [r*S, (r+1)*S) of every rank's flat
     gradient (the same bytes a ring reduce-scatter moves) and every rank's
     persistent-group gradient (the bytes of their all-gather).  The sum runs in
     the fused kernel, in fixed rank order in binary32, so the result is bit
     for bit the one-GPU emulation's (a collective that sums in bf16 in its
     own order would not be).
  2. the fused AdamW step on rank r's fp32 master/m/v shard and its bf16
     parameter shard (zero3_step over flat [r*S, (r+1)*S), gradients read
     from the received slices), and the persistent group's DDP-style update
     on its replicated copy;
  3. the parameter all-gather: every rank's updated bf16 shard into every
     rank's flat buffer `full`.

Allocation and call plumbing only: the arithmetic of step 2 is the C-ABI
library's (or, for CPU tests, a step function the caller passes in).  No
multicast or peer-memory access is used; the collectives are the library's.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch
import torch.distributed as dist

from . import zero3


class ShardedRank:
    """Rank `rank` of a world of N_d = plan.info.n_ranks processes.

    Buffers (on `device`; bf16 data is kept in torch.bfloat16 tensors, which
    every backend moves byte for byte).  S8 and P8 are S and psi_s rounded up
    to a multiple of 8 elements, so every row below starts 16-byte aligned,
    as the library's gradient pointers must:
      grad    [psi_pad + psi_s]    this rank's local gradient: flat, then the
                                   persistent group (filled by the caller)
      send    [N_d, S8 + P8]       row q: slice q of the flat gradient, then
                                   the persistent group's gradient
      recv    [N_d, S8 + P8]       row q: slice r of rank q's flat gradient,
                                   then rank q's persistent-group gradient
      master, m, v [S] fp32; sparam [S] bf16: rank r's shard
      full    [psi_pad] bf16       the all-gathered flat parameters
      pmaster, pm, pv [psi_s] fp32; pparam [psi_s] bf16: the persistent
                                   group, replicated on every rank
    Sending the persistent gradients in every row moves the same bytes as
    their all-gather and puts them at one offset (S8) from each rank's slice,
    so the local step is a single fused launch.
    """

    def __init__(self, plan: zero3.Plan, hp, rank: int, device="cuda",
                 group: Optional[dist.ProcessGroup] = None,
                 local_step: Optional[Callable[["ShardedRank", int], None]] = None):
        info = plan.info
        self.plan, self.hp, self.rank = plan, hp, rank
        self.nd, self.S = info.n_ranks, info.shard_len
        self.psi_pad, self.psi_s = info.psi_pad, info.psi_s
        self.S8 = (self.S + 7) // 8 * 8
        self.P8 = (self.psi_s + 7) // 8 * 8
        self.group = group
        self.dev = torch.device(device)
        bf, f32 = torch.bfloat16, torch.float32
        z = lambda n, dt: torch.zeros(n, dtype=dt, device=self.dev)
        self.grad = z(self.psi_pad + self.psi_s, bf)
        self.send = torch.zeros(self.nd, self.S8 + self.P8, dtype=bf, device=self.dev)
        self.recv = torch.zeros(self.nd, self.S8 + self.P8, dtype=bf, device=self.dev)
        self.master, self.m, self.v = z(self.S, f32), z(self.S, f32), z(self.S, f32)
        self.sparam, self.full = z(self.S, bf), z(self.psi_pad, bf)
        self.pmaster, self.pm, self.pv = z(self.psi_s, f32), z(self.psi_s, f32), z(self.psi_s, f32)
        self.pparam = z(self.psi_s, bf)
        self.local_step = local_step or ShardedRank.fused_step

    def slice_of(self, q: int) -> torch.Tensor:
        """The received slice r of rank q's flat gradient (S elements)."""
        return self.recv[q, :self.S]

    def persist_of(self, q: int) -> torch.Tensor:
        """Rank q's persistent-group gradient (psi_s elements)."""
        return self.recv[q, self.S8:self.S8 + self.psi_s]

    # ------------------------------------------------------------ the step
    def exchange(self) -> None:
        """Step 1's communication, one all-to-all: row q of recv holds slice
        r of rank q's flat gradient and rank q's persistent gradient."""
        nd, S, S8 = self.nd, self.S, self.S8
        self.send[:, :S].copy_(self.grad[:self.psi_pad].view(nd, S))
        if self.psi_s > 0:
            self.send[:, S8:S8 + self.psi_s].copy_(
                self.grad[self.psi_pad:].unsqueeze(0).expand(nd, self.psi_s))
        dist.all_to_all_single(self.recv.view(-1), self.send.view(-1), group=self.group)

    def gather(self) -> None:
        """Step 3: every rank's bf16 shard into every rank's `full`."""
        if self.psi_pad > 0:
            dist.all_gather_into_tensor(self.full, self.sparam, group=self.group)

    def step(self, t: int) -> None:
        self.exchange()
        self.local_step(self, t)
        self.gather()

    # ------------------------------------------------------------ the CUDA step
    def fused_step(self, t: int) -> None:
        """Step 2 through the C ABI on this rank's GPU: the fused kernel over
        flat [r*S, (r+1)*S), whose gradients are the received slices
        (grads[q] + (f - r*S) for flat f), and the persistent group."""
        r, nd = self.rank, self.nd
        lo, hi = r * self.S, (r + 1) * self.S
        only = lambda x: [x.data_ptr() if q == r else 0 for q in range(nd)]
        # the persistent gradients sit S8 elements after each slice: one launch
        ps = zero3.persist_state([self.persist_of(q).data_ptr() for q in range(nd)],
                                 self.pmaster.data_ptr(), self.pm.data_ptr(), self.pv.data_ptr(),
                                 self.pparam.data_ptr()) if self.psi_s > 0 else None
        stream = torch.cuda.current_stream(self.dev).cuda_stream
        zero3.zero3_step(self.plan, self.hp, t, [self.slice_of(q).data_ptr() for q in range(nd)],
                         lo, only(self.master), only(self.m), only(self.v), only(self.sparam),
                         self.full.data_ptr(), ps, lo, hi, stream)

    def cast_params(self) -> None:
        """bf16 shard, this rank's part of `full` and the persistent params
        from the fp32 masters (initialisation, after loading states)."""
        r, nd = self.rank, self.nd
        only = lambda x: [x.data_ptr() if q == r else 0 for q in range(nd)]
        ps = zero3.persist_state([0] * nd, self.pmaster.data_ptr(), self.pm.data_ptr(),
                                 self.pv.data_ptr(), self.pparam.data_ptr()) \
            if self.psi_s > 0 else None
        stream = torch.cuda.current_stream(self.dev).cuda_stream
        zero3.zero3_cast_params(self.plan, only(self.master), only(self.sparam),
                                self.full.data_ptr(), ps, r * self.S, (r + 1) * self.S, stream)
