"""N_d virtual data-parallel ranks laid out in one GPU's HBM.

Allocation and call plumbing only: PyTorch allocates the buffers, the seeded
device generator fills the inputs, and every step of the path is a call into
libzero3 through the `zero3` binding.

Layout (all separate allocations, each 512-byte aligned by the allocator):
  gbufs[c][q]   bf16  rank q's local gradient buffer for flat range chunk c
                      (chunk c = [lo_c, hi_c)); the first chunk's buffer also
                      holds the persistent group's gradients after the flat
                      ones (at the next 16-byte boundary), so one fused launch
                      covers both
  grads[c][q]   view  the flat part: index f at grads[c][q][f - lo_c]
  pgrads[q]     view  rank q's local gradient of the persistent group (psi_s)
  master/m/v[r] fp32  rank r's optimizer-state shard (S), only for state ranks
  sparam[r]     bf16  rank r's parameter shard (S), every rank
  full          bf16  the flat all-gathered parameter buffer (psi_pad)
  pmaster/pm/pv fp32, pparam bf16: the one resident copy of the persistent group
  out           bf16  the submodule gather buffer (largest submodule)
  arena         bf16  the gather buffers of one all-gather bucket (allocated on
                      first use): each submodule of the bucket at its own
                      16-byte aligned offset
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import synth_device, zero3
from .workloads import (STREAM_GRAD, STREAM_GRAD_PERSIST, STREAM_MASTER,
                        STREAM_MASTER_PERSIST, Workload)


def _ptr(t: Optional[torch.Tensor]) -> int:
    return t.data_ptr() if t is not None else 0


# Sentinels of the guard bands (bit patterns; NaN payloads for the floats).
_SENTINEL = {torch.float32: 0x7FC0DEAD, torch.bfloat16: 0x7FAD, torch.int8: 0x5A}
_INT_VIEW = {torch.float32: torch.int32, torch.bfloat16: torch.int16, torch.int8: torch.int8}


class Emulation:
    def __init__(self, w: Workload, device: str = "cuda", state_ranks: Optional[Sequence[int]] = None,
                 bucketed: bool = False, stream: Optional[torch.cuda.Stream] = None,
                 alloc_grads: bool = True, guard: int = 0):
        """guard > 0 surrounds every buffer with `guard` sentinel elements on
        each side (guard-band canaries); check_guards() reports any band a
        call has written into."""
        self.w = w
        self.dev = torch.device(device)
        self.guard = guard
        self._guarded = []
        self.plan = zero3.Plan(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
        info = self.plan.info
        self.nd = w.n_ranks
        self.S = info.shard_len
        self.psi_p, self.psi_pad, self.psi_s = info.psi_p, info.psi_pad, info.psi_s
        self.state_ranks = list(range(self.nd)) if state_ranks is None else sorted(state_ranks)
        self.hp = zero3.hparams(**w.hparams)
        self.stream = stream
        # flat range whose owners hold optimizer state on this device
        lo = min(self.state_ranks) * self.S
        hi = (max(self.state_ranks) + 1) * self.S
        assert self.state_ranks == list(range(min(self.state_ranks), max(self.state_ranks) + 1)), \
            "state ranks must be consecutive"
        if bucketed:
            cuts = sorted({lo, hi} | {b for b in range(0, self.psi_pad, w.bucket) if lo < b < hi})
            self.chunks = list(zip(cuts[:-1], cuts[1:]))
        else:
            self.chunks = [(lo, hi)] if hi > lo else []
        bf, f32 = torch.bfloat16, torch.float32
        A = self.alloc
        self.gbufs: List[List[torch.Tensor]] = []
        self.grads: List[List[torch.Tensor]] = []
        self.pgrads: List[torch.Tensor] = []
        if alloc_grads:
            for c, (a, b) in enumerate(self.chunks):
                n = b - a
                tail = (n + 7) // 8 * 8 + self.psi_s if c == 0 else n
                bufs = [A(tail, bf) for _ in range(self.nd)]
                self.gbufs.append(bufs)
                self.grads.append([x[:n] for x in bufs])
                if c == 0:
                    o = (n + 7) // 8 * 8
                    self.pgrads = [x[o:o + self.psi_s] for x in bufs]
        if not self.pgrads:
            self.pgrads = [A(self.psi_s, bf) for _ in range(self.nd)]
        self.master: List[Optional[torch.Tensor]] = [None] * self.nd
        self.m: List[Optional[torch.Tensor]] = [None] * self.nd
        self.v: List[Optional[torch.Tensor]] = [None] * self.nd
        for r in self.state_ranks:
            self.master[r] = A(self.S, f32)
            self.m[r] = A(self.S, f32, zero=True)
            self.v[r] = A(self.S, f32, zero=True)
        self.sparam = [A(self.S, bf) for _ in range(self.nd)]
        self.full = A(self.psi_pad, bf, zero=True)
        self.pmaster = A(self.psi_s, f32)
        self.pm = A(self.psi_s, f32, zero=True)
        self.pv = A(self.psi_s, f32, zero=True)
        self.pparam = A(self.psi_s, bf)
        self.max_sub = max([self.plan.submodule(k)[1] for k in range(info.n_submodules)] + [0])
        self.out = A(max(self.max_sub, 1), bf)
        self.arena: Optional[torch.Tensor] = None
        self._buckets: dict = {}
        self.persist = zero3.persist_state([_ptr(g) for g in self.pgrads], _ptr(self.pmaster),
                                           _ptr(self.pm), _ptr(self.pv), _ptr(self.pparam))

    # ------------------------------------------------------------ plumbing
    def alloc(self, n: int, dtype, zero: bool = False) -> torch.Tensor:
        """A device buffer of n elements (16-byte aligned); with guard bands
        when the emulation was created with guard > 0."""
        g = self.guard
        if g <= 0:
            return (torch.zeros if zero else torch.empty)(n, dtype=dtype, device=self.dev)
        base = torch.empty(n + 2 * g, dtype=dtype, device=self.dev)
        base.view(_INT_VIEW[dtype]).fill_(_SENTINEL[dtype])
        view = base[g:g + n]
        if zero:
            view.zero_()
        self._guarded.append((base, g, n, dtype))
        return view

    def check_guards(self) -> List[str]:
        """Names of the buffers whose guard bands were written."""
        bad = []
        for i, (base, g, n, dtype) in enumerate(self._guarded):
            iv = base.view(_INT_VIEW[dtype])
            want = _SENTINEL[dtype]
            if not (bool((iv[:g] == want).all()) and bool((iv[g + n:] == want).all())):
                bad.append(f"buffer {i} ({dtype}, {n} elements)")
        return bad

    @property
    def sid(self) -> int:
        s = self.stream if self.stream is not None else torch.cuda.current_stream(self.dev)
        return s.cuda_stream

    def ptrs(self, xs) -> List[int]:
        return [_ptr(x) for x in xs]

    # ------------------------------------------------------------ inputs
    def init_params(self) -> None:
        """fp32 masters from the generator (padding zero), m = v = 0, then the
        bf16 shards, the full buffer and the persistent params via
        zero3_cast_params.  Shards of ranks without state are cast from a
        temporary master."""
        w = self.w
        for r in range(self.nd):
            tmp = self.master[r] if self.master[r] is not None else \
                torch.empty(self.S, dtype=torch.float32, device=self.dev)
            n = max(0, min(self.S, self.psi_p - r * self.S))
            if self.S > n:
                tmp[n:].zero_()
            synth_device.normal(_ptr(tmp), n, seed=w.seed, stream_id=STREAM_MASTER, step=0, rank=0,
                                index0=r * self.S, sigma=w.master_sigma, bf16=False,
                                cuda_stream=self.sid)
            masters = [0] * self.nd
            sparams = [0] * self.nd
            masters[r] = _ptr(tmp)
            sparams[r] = _ptr(self.sparam[r])
            zero3.zero3_cast_params(self.plan, masters, sparams, _ptr(self.full), None,
                                    r * self.S, (r + 1) * self.S, self.sid)
        synth_device.normal(_ptr(self.pmaster), self.psi_s, seed=w.seed,
                            stream_id=STREAM_MASTER_PERSIST, step=0, rank=0, index0=0,
                            sigma=w.master_sigma, bf16=False, cuda_stream=self.sid)
        zero3.zero3_cast_params(self.plan, None, None, 0, self.persist, 0, 0, self.sid)

    def fill_grads(self, step: int) -> None:
        """Every rank's local gradient for `step` from the generator; the
        padding [psi_p, psi_pad) is zero."""
        w = self.w
        for (a, b), G in zip(self.chunks, self.grads):
            n = max(0, min(b, self.psi_p) - a)
            for q in range(self.nd):
                if b - a > n:
                    G[q][n:].zero_()
                synth_device.normal(_ptr(G[q]), n, seed=w.seed, stream_id=STREAM_GRAD, step=step,
                                    rank=q, index0=a, sigma=w.grad_sigma, outlier_p=w.outlier_p,
                                    outlier_sigma=w.outlier_sigma, cuda_stream=self.sid)
        for q in range(self.nd):
            synth_device.normal(_ptr(self.pgrads[q]), self.psi_s, seed=w.seed,
                                stream_id=STREAM_GRAD_PERSIST, step=step, rank=q, index0=0,
                                sigma=w.grad_sigma, outlier_p=w.outlier_p,
                                outlier_sigma=w.outlier_sigma, cuda_stream=self.sid)

    # ------------------------------------------------------------ the path
    def step(self, t: int, with_persistent: bool = True) -> None:
        """The fused ZeRO-3 step over every chunk (one launch per chunk) and
        the persistent group."""
        for c, ((a, b), G) in enumerate(zip(self.chunks, self.grads)):
            zero3.zero3_step(self.plan, self.hp, t, self.ptrs(G), a, self.ptrs(self.master),
                             self.ptrs(self.m), self.ptrs(self.v), self.ptrs(self.sparam),
                             _ptr(self.full), self.persist if (with_persistent and c == 0) else None,
                             a, b, self.sid)
        if with_persistent and not self.chunks:
            zero3.zero3_persistent_step(self.plan, self.hp, t, self.persist, self.sid)

    def fetch(self, k: int) -> None:
        zero3.zero3_fetch_submodule(self.plan, k, self.ptrs(self.sparam), _ptr(self.pparam),
                                    _ptr(self.out), self.sid)

    def release(self, k: int) -> None:
        zero3.zero3_release_submodule(self.plan, k)

    def gather_buckets(self, bucket: int) -> List[List[int]]:
        """Consecutive submodules grouped into buckets of at most `bucket`
        elements (a larger submodule forms a bucket of its own)."""
        if bucket in self._buckets:
            return self._buckets[bucket]
        groups: List[List[int]] = []
        cur: List[int] = []
        size = 0
        for k in range(self.plan.info.n_submodules):
            n = self.plan.submodule(k)[1]
            if cur and size + n > bucket:
                groups.append(cur)
                cur, size = [], 0
            cur.append(k)
            size += n
        if cur:
            groups.append(cur)
        self._buckets[bucket] = groups
        return groups

    def bucket_outputs(self, ks: Sequence[int]) -> List[int]:
        """Device pointers of the gather buffers of submodules ks, each at a
        16-byte aligned offset of the arena (grown to the largest bucket)."""
        sizes = [(self.plan.submodule(k)[1] + 7) // 8 * 8 for k in ks]
        need = max(sum(sizes), 8)
        if self.arena is None or self.arena.numel() < need:
            self.arena = self.alloc(need, torch.bfloat16)
        base = self.arena.data_ptr()
        outs, off = [], 0
        for n in sizes:
            outs.append(base + 2 * off)
            off += n
        return outs

    def fetch_many(self, ks: Sequence[int]) -> List[int]:
        """One zero3_fetch_submodules call for submodules ks; returns their
        gather buffers."""
        outs = self.bucket_outputs(ks)
        zero3.zero3_fetch_submodules(self.plan, list(ks), self.ptrs(self.sparam),
                                     _ptr(self.pparam), outs, self.sid)
        return outs

    def forward_backward_gathers(self, bucket: int = 0) -> None:
        """Gather every submodule before its forward (list order) and again
        before its backward (reverse order), releasing after each use.  With
        bucket > 0 consecutive submodules of up to `bucket` elements are
        gathered together (one zero3_fetch_submodules call per bucket),
        forward in list order and backward in reverse."""
        n = self.plan.info.n_submodules
        if bucket > 0:
            groups = self.gather_buckets(bucket)
            self.bucket_outputs(max(groups, key=lambda g: sum(
                (self.plan.submodule(k)[1] + 7) // 8 * 8 for k in g)) if groups else [])
            for ks in groups + [list(reversed(g)) for g in reversed(groups)]:
                self.fetch_many(ks)
                for k in ks:
                    self.release(k)
            return
        for k in range(n):
            self.fetch(k)
            self.release(k)
        for k in reversed(range(n)):
            self.fetch(k)
            self.release(k)

    def full_step(self, t: int) -> None:
        self.forward_backward_gathers()
        self.step(t)

    # ------------------------------------------------------------ accounting
    def step_bytes(self) -> dict:
        """Algorithmic HBM bytes of one full step (fused step + persistent +
        two gathers of every submodule)."""
        nd = self.nd
        n_flat = sum(b - a for a, b in self.chunks)
        fused = n_flat * (2 * nd + 24 + 2 + 2)
        persist = self.psi_s * (2 * nd + 24 + 2)
        gathers = 2 * sum(self.plan.submodule(k)[1] for k in range(self.plan.info.n_submodules)) * 4
        return dict(fused=fused, persistent=persist, gathers=gathers,
                    total=fused + persist + gathers, flat_elems=n_flat)
