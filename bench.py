"""Benchmark of the ZeRO-3 hot path: one step = a forward and a backward
gather of every submodule plus the fused reduce-scatter/AdamW/cast/all-gather
step over every virtual rank and the persistent group.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decoder_1p3b|gpt2_small|llama_7b_rank0]

Prints one JSON line (rank 0).  N > 1 runs one replica of the workload per
GPU (the emulated ranks live inside each GPU; there is no inter-GPU step),
launched by torch.distributed.run; value is the params of all replicas per
second (weak scaling).  --impl reference times the CPU oracle on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused ZeRO-3 step params/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
PROFILE = os.path.join(ROOT, "profiles", "zero3_step_fused_decoder_1p3b.md")

WORKLOADS = {
    # name: (factory, state ranks, bucketed, description)
    "decoder_1p3b": ("decoder_1p3b", None, False,
                     "1.3B GPT-style decoder (24L, d=2048, vocab 50257), N_d=8 virtual ranks, "
                     "full emulation in one HBM"),
    "gpt2_small": ("gpt2_small", None, False,
                   "GPT-2-small list (12L, d=768, vocab 50257), N_d=4 virtual ranks"),
    "ragged": ("ragged", None, False,
               "Ragged list: 2000 tensors, log-uniform sizes (30% below 1e5), N_d=7 virtual ranks"),
    "llama_7b_full": ("llama_7b_full", None, True,
                      "Llama-7B list, all N_d=8 ranks emulated in one HBM (~216 GB), "
                      "one fused launch per 5e8-element bucket"),
    "llama_7b_rank0": ("llama_7b_rank0", [0], True,
                       "Llama-7B list (32L, d=4096, SwiGLU 11008, vocab 32000), rank-0 view at "
                       "N_d=8: rank 0's state resident, gradients per 5e8-element bucket"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decoder_1p3b")
    ap.add_argument("--n-ranks", type=int, default=None,
                    help="override the workload's N_d (small profiling cases)")
    ap.add_argument("--stage", type=int, choices=[2, 3], default=3,
                    help="3: ZeRO-3 step (default); 2: the ZeRO-1/2 step (full parameters on "
                         "every rank, no submodule gathers)")
    ap.add_argument("--coordinator", action="store_true",
                    help="measure the prefetching coordinator: forward/backward gathers "
                         "interleaved with a GEMM per submodule, prefetch on vs off")
    ap.add_argument("--tokens", type=int, default=4096,
                    help="rows of the stand-in activation for --coordinator")
    ap.add_argument("--qwz", action="store_true",
                    help="ZeRO++ qwZ: the fused step emits int8 codes + block scales and the "
                         "all-gather dequantizes them into the full buffer")
    ap.add_argument("--qwz-bits", type=int, choices=[8, 4], default=8)
    ap.add_argument("--unfused", action="store_true",
                    help="ablation: reduce-scatter (fp32 shard gradient), AdamW and all-gather "
                         "as three launches, each timed")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profile_traffic(kernels_sha: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu
    summary, if it was captured on the current kernel source."""
    if not os.path.exists(PROFILE):
        return None
    txt = open(PROFILE).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(kernels\.cu sha256 ([0-9a-f]+)\)", txt)
    if not m or m.group(2) != kernels_sha:
        return None
    return float(m.group(1))


def kernels_sha() -> str:
    p = os.path.join(ROOT, "zero_sharded_optimizer_shard_gb300", "csrc", "kernels.cu")
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples every 50 ms; stop() keeps the samples taken inside
    the timed window [t0, t1] (host clock)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float):
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]),
                             [parts[6 + k].lower().startswith("active") for k in range(4)]))
            except ValueError:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:  # timed region shorter than the sampling interval
            inside = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1]
            window = "timed region +-100 ms"
        reasons = sorted({n for r in inside for n, a in zip(self.NAMES, r[4]) if a})
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "power_w_max": max(r[3] for r in inside) if inside else None,
                "samples": len(inside), "window": window, "reasons": reasons}


def make_workload(args):
    from zero_sharded_optimizer_shard_gb300 import workloads as W
    fac = WORKLOADS[args.workload][0]
    w = W.llama_7b(rank0_view=(fac == "llama_7b_rank0")) if fac.startswith("llama_7b") \
        else getattr(W, fac)()
    if args.n_ranks:
        w.n_ranks = args.n_ranks
    if args.stage == 2:
        w.threshold = 0  # the persistence threshold is a stage-3 setting
    return w


def step_config(args, w, world, psi_pad, psi_s, n_flat, sub_numels):
    """The `config` object of the step benchmark, from the partition's sizes
    alone, so that both arms (GPU path and CPU oracle) report the same one.
    Bytes per step: the fused step (2*N_d + 28 per flat element), the
    persistent group (2*N_d + 26) and two gathers of every submodule (4)."""
    nd = w.n_ranks
    total = n_flat * (2 * nd + 28) + psi_s * (2 * nd + 26) + 2 * sum(sub_numels) * 4
    desc = WORKLOADS[args.workload][3]
    if args.n_ranks:
        desc += f" (N_d overridden to {nd})"
    params = w.psi if WORKLOADS[args.workload][1] is None else n_flat + psi_s
    return {
        "workload": desc, "name": args.workload, "n_ranks": nd,
        "params": params, "psi_pad": psi_pad, "psi_s": psi_s,
        "bytes_per_step": total,
        "step": "forward + backward gather of every submodule, fused step, persistent group",
        "l2": f"inputs larger than L2 ({total / 1e9:.1f} GB touched per step)",
        "grads": "generated once on the device before timing, reused by every step",
        "parallelism": f"{world} replica(s) x {nd} emulated ranks",
    }


def cpu_oracle_rate(w, budget_s: float = 15.0):
    """The CPU oracle, as it stands, on a bounded contiguous sample of rank
    0's shard: all N_d ranks' gradients for the sample, the reduce, AdamW and
    bf16 cast.  Returns (params/s, description)."""
    import numpy as np

    import oracle as O
    from zero_sharded_optimizer_shard_gb300 import synth, workloads as W

    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    rng_n = 1 << 20
    idx = np.arange(rng_n, dtype=np.int64)
    grads = [synth.normal_bf16(w.seed, W.STREAM_GRAD, 1, q, idx, w.grad_sigma, w.outlier_p,
                               w.outlier_sigma) for q in range(plan.n_ranks)]
    p = synth.normal_f32(w.seed, W.STREAM_MASTER, 0, 0, idx, w.master_sigma)
    m = np.zeros_like(p)
    v = np.zeros_like(p)

    def one(t, p, m, v):
        sc = O.adamw_scalars(w.hparams, t, plan.n_ranks)
        g = O.reduce_sum(grads, sc["inv_nd"])
        p, m, v = O.adamw_update(g, p, m, v, sc)
        return p, m, v, O.cast_bf16(p)

    t0 = time.perf_counter()
    p, m, v, _ = one(1, p, m, v)
    dt1 = time.perf_counter() - t0
    reps = max(1, int(budget_s / max(dt1, 1e-3)))
    t0 = time.perf_counter()
    for t in range(2, 2 + reps):
        p, m, v, _ = one(t, p, m, v)
    dt = time.perf_counter() - t0
    rate = rng_n * reps / dt
    return rate, (f"{rng_n} consecutive elements of rank 0's shard, all {plan.n_ranks} ranks' "
                  f"gradients, {reps} steps (numpy, one thread)"), dt


def run_reference(args):
    import numpy as np  # noqa: F401
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle as O
    w = make_workload(args)
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    n_flat = plan.psi_pad if WORKLOADS[args.workload][1] is None else plan.shard_len
    config = step_config(args, w, args.gpus, plan.psi_pad, plan.psi_s, n_flat,
                         [plan.submodule_numel(k) for k in range(plan.n_submodules)])
    budget = 4.0
    rates = []
    desc = None
    for i in range(args.warmup + args.steps):
        r, desc, _ = cpu_oracle_rate(make_workload(args), budget_s=budget)
        if i >= args.warmup:
            rates.append(r)
    value = sum(rates) / len(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # the oracle's time for one whole step of the workload, extrapolated
        # from the sample's rate
        "ms_per_step": config["params"] / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def reduce_max(value: float, device) -> float:
    """Max of a per-rank value over the process group (barrier included)."""
    import torch
    import torch.distributed as dist
    x = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return float(x.item())


def replica_throughput(world: int, params_per_replica: int, ms_per_step: float) -> float:
    """Weak scaling: every replica processes its own copy of the workload, so
    the job's params/s is world x params / the slowest rank's step time."""
    return world * params_per_replica / (ms_per_step / 1e3)


def launches_per_step(e) -> int:
    """Kernel launches of one full step, counted from the plan: the fused
    kernel once per gradient chunk, the persistent group once, and each
    submodule gather ceil(pieces / 64) times, twice (forward, backward)."""
    import math
    n = 0
    for k in range(e.plan.info.n_submodules):
        pieces = 0
        for t, sub in enumerate(e.w.submodule_of):
            if sub != k or e.w.numels[t] == 0:
                continue
            ti = e.plan.tensor(t)
            pieces += 1 if ti.persistent else ti.n_segments
        n += 2 * math.ceil(pieces / 64)
    return n + len(e.chunks) + (1 if e.psi_s > 0 else 0)


def setup_single(args, stream=None, **emu_kw):
    """Build the library, create the workload's emulation on cuda:0 and fill
    its inputs (shared by the single-GPU measurement modes)."""
    import torch
    from zero_sharded_optimizer_shard_gb300 import build as b
    b.build_all(quiet=True)
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation
    torch.cuda.set_device(0)
    fac, state_ranks, bucketed, desc = WORKLOADS[args.workload]
    w = make_workload(args)
    if args.n_ranks:
        desc += f" (N_d overridden to {w.n_ranks})"
    stream = stream or torch.cuda.Stream()
    kw = dict(state_ranks=state_ranks, bucketed=bucketed)
    kw.update(emu_kw)
    e = Emulation(w, stream=stream, **kw)
    with torch.cuda.stream(stream):
        e.init_params()
        e.fill_grads(1)
    torch.cuda.synchronize()
    return w, e, stream, desc


def run_stage12(args):
    """The ZeRO-1/2 step: every rank keeps full bf16 parameters, so a step is
    the fused reduce-scatter + AdamW + all-gather into all N_d copies."""
    import torch
    from zero_sharded_optimizer_shard_gb300 import zero3
    if WORKLOADS[args.workload][1] is not None:
        raise SystemExit("--stage 2 needs a full emulation workload")
    w, e, stream, desc = setup_single(args, bucketed=False)
    with torch.cuda.stream(stream):
        params = [e.full.clone() for _ in range(w.n_ranks)]
    e.sparam = e.full = None  # stage 1/2 keeps no separate shard or gathered buffer
    torch.cuda.synchronize()
    pp = [x.data_ptr() for x in params]
    lo, hi = e.chunks[0]

    def step(t):
        zero3.zero3_step_stage12(e.plan, e.hp, t, e.ptrs(e.grads[0]), lo, e.ptrs(e.master),
                                 e.ptrs(e.m), e.ptrs(e.v), pp, lo, hi, e.sid)

    t = 0
    for _ in range(args.warmup):
        t += 1
        step(t)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.5)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    tw0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        t += 1
        step(t)
    end.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    ms = start.elapsed_time(end) / args.steps
    clk = clocks.stop(tw0, tw1)
    n_el = hi - lo
    bpe = 4 * w.n_ranks + 24
    peak, peak_kind = peaks()
    achieved = n_el * bpe / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": METRIC, "value": w.psi / (ms / 1e3), "unit": "params/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": desc + ", ZeRO-1/2 step (full bf16 parameters on every rank)",
                   "name": args.workload, "stage": "1/2", "n_ranks": w.n_ranks, "params": w.psi,
                   "bytes_per_elem": bpe},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": None,
                     "kernel": "stream_kernel<kFusedRep, N_d> (zero3_step_stage12)"},
        "gpu_launches": args.steps, "clocks": clk, "cpu_baseline": None, "e2e": None}))
    return 0


def run_coordinator(args):
    """Forward then backward over the submodules, each gathered through the
    prefetching coordinator and consumed by bf16 GEMMs (one in forward, two
    in backward) that stand in for the model's compute, then the fused
    optimizer step.  Timed three ways on the same buffers: prefetch on,
    prefetch off (every gather on demand), and the GEMMs alone (no gathers);
    the difference off - on is the gather time the prefetch hides."""
    import torch
    from zero_sharded_optimizer_shard_gb300 import zero3
    if WORKLOADS[args.workload][1] is not None:
        raise SystemExit("--coordinator needs a full emulation workload")
    w, e, compute, desc = setup_single(args, bucketed=False)
    prefetch = torch.cuda.Stream()
    plan = e.plan
    n_sub = plan.info.n_submodules
    sizes = [plan.submodule(k)[1] for k in range(n_sub)]
    trace = list(range(n_sub)) + list(reversed(range(n_sub)))
    arena_elems = (3 * max(sizes) + 7) // 8 * 8
    arena = torch.empty(arena_elems, dtype=torch.bfloat16, device="cuda")
    width = 1024
    X = torch.randn(args.tokens, width, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(args.tokens, max(sizes) // width + 1, dtype=torch.bfloat16, device="cuda")
    dX = torch.empty(args.tokens, width, dtype=torch.bfloat16, device="cuda")
    Wfix = torch.randn(arena_elems, dtype=torch.bfloat16, device="cuda")

    def gemms(buf, off, k, backward):
        cols = sizes[k] // width
        if cols == 0:
            return
        Wv = buf[off:off + cols * width].view(width, cols)
        torch.matmul(X, Wv, out=Y[:, :cols])
        if backward:
            torch.matmul(Y[:, :cols], Wv.t(), out=dX)

    def one_step(co, t):
        for i, k in enumerate(trace):
            if co is None:
                with torch.cuda.stream(compute):
                    gemms(Wfix, 0, k, i >= n_sub)
                continue
            ptr = co.fetch(k)
            with torch.cuda.stream(compute):
                gemms(arena, (ptr - arena.data_ptr()) // 2, k, i >= n_sub)
            co.release(k)
        e.step(t)
        if co is not None:
            co.next_step()

    results = {}
    t = 0
    for mode, bucket in (("prefetch", w.bucket), ("on_demand", 0), ("gemm_only", None)):
        co = None
        if bucket is not None:
            co = zero3.Coordinator(plan, trace, e.ptrs(e.sparam), e.pparam.data_ptr(),
                                   arena.data_ptr(), arena_elems, prefetch_bucket_size=bucket,
                                   max_live_parameters=arena_elems,
                                   max_reuse_distance=10**9, compute_stream=compute.cuda_stream,
                                   prefetch_stream=prefetch.cuda_stream)
        for _ in range(args.warmup):
            t += 1
            one_step(co, t)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(compute)
        for _ in range(args.steps):
            t += 1
            one_step(co, t)
        s1.record(compute)
        torch.cuda.synchronize()
        results[mode] = {"ms_per_step": s0.elapsed_time(s1) / args.steps}
        if co is not None:
            results[mode]["stats"] = co.stats()
        del co
    hidden = results["on_demand"]["ms_per_step"] - results["prefetch"]["ms_per_step"]
    exposed = results["on_demand"]["ms_per_step"] - results["gemm_only"]["ms_per_step"]
    print(json.dumps({
        "metric": "ZeRO-3 forward/backward step with submodule gathers, prefetch on vs off",
        "value": results["prefetch"]["ms_per_step"], "unit": "ms/step", "higher_is_better": False,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "data": "synthetic",
        "config": {"workload": desc, "tokens": args.tokens,
                   "compute": f"bf16 GEMM [{args.tokens} x {width}] x [{width} x numel/{width}] "
                              "per submodule (2 in backward)",
                   "arena_elems": arena_elems, "prefetch_bucket_size": w.bucket},
        "modes": results,
        "gather_ms_hidden": hidden,
        "gather_ms_exposed_without_prefetch": exposed,
        "hidden_fraction": hidden / exposed if exposed > 0 else None}))
    return 0


def run_qwz(args):
    """The qwZ step: fused reduce-scatter + AdamW + bf16 shard + int8 block
    quantization, then the dequantizing all-gather into the full buffer."""
    import torch
    from zero_sharded_optimizer_shard_gb300 import zero3
    if WORKLOADS[args.workload][1] is not None:
        raise SystemExit("--qwz needs a full emulation workload")
    w, e, stream, desc = setup_single(args, bucketed=False)
    nb = -(-e.S // 256)
    with torch.cuda.stream(stream):
        codes = [torch.empty(-(-e.S * args.qwz_bits // 8), dtype=torch.int8, device="cuda")
                 for _ in range(e.nd)]
        scales = [torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(e.nd)]
    torch.cuda.synchronize()
    cp, sp = e.ptrs(codes), e.ptrs(scales)
    lo, hi = e.chunks[0]
    ev = []

    def step(t, timed):
        a0, a1, a2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a0.record(stream)
        zero3.zero3_step_qwz(e.plan, e.hp, t, e.ptrs(e.grads[0]), lo, e.ptrs(e.master), e.ptrs(e.m),
                             e.ptrs(e.v), e.ptrs(e.sparam), cp, sp, None, lo, hi, e.sid,
                             bits=args.qwz_bits)
        a1.record(stream)
        zero3.zero3_allgather_qwz(e.plan, cp, sp, e.full.data_ptr(), lo, hi, e.sid,
                                  bits=args.qwz_bits)
        a2.record(stream)
        zero3.zero3_persistent_step(e.plan, e.hp, t, e.persist, e.sid)
        if timed:
            ev.append((a0, a1, a2))

    t = 0
    for _ in range(args.warmup):
        t += 1
        step(t, False)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.5)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    tw0 = time.time()
    s0.record(stream)
    for _ in range(args.steps):
        t += 1
        step(t, True)
    s1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    clk = clocks.stop(tw0, tw1)
    ms = s0.elapsed_time(s1) / args.steps
    fused_ms = statistics.mean(a.elapsed_time(b_) for a, b_, _ in ev)
    gather_ms = statistics.mean(b_.elapsed_time(c) for _, b_, c in ev)
    n = hi - lo
    cb = args.qwz_bits / 8
    fused_bytes = n * (2 * w.n_ranks + 24 + 2 + cb) + e.nd * nb * 4
    gather_bytes = n * (cb + 2) + e.nd * nb * 4
    peak, peak_kind = peaks()
    ach = fused_bytes / (fused_ms / 1e3) / 1e9
    print(json.dumps({
        "metric": METRIC, "value": w.psi / (ms / 1e3), "unit": "params/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": desc + f", qwZ int{args.qwz_bits} all-gather (block 256)",
                   "name": args.workload,
                   "n_ranks": w.n_ranks, "params": w.psi},
        "fused_qwz": {"ms_per_launch": fused_ms, "bytes_per_launch": fused_bytes,
                      "gbs": ach, "frac": ach / peak},
        "allgather_qwz": {"ms_per_launch": gather_ms, "bytes_per_launch": gather_bytes,
                          "gbs": gather_bytes / (gather_ms / 1e3) / 1e9},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                     "frac": ach / peak, "peak_kind": peak_kind, "traffic": None,
                     "kernel": "stream_kernel<kFusedQ, N_d> (zero3_step_qwz)"},
        "gpu_launches": 3 * args.steps, "clocks": clk, "cpu_baseline": None, "e2e": None}))
    return 0


def run_unfused(args):
    """Ablation: the same step as three launches (what fusion saves)."""
    import torch
    from zero_sharded_optimizer_shard_gb300 import zero3
    if WORKLOADS[args.workload][1] is not None:
        raise SystemExit("--unfused needs a full emulation workload")
    w, e, stream, desc = setup_single(args, bucketed=False)
    with torch.cuda.stream(stream):
        sg = [torch.empty(e.S, dtype=torch.float32, device="cuda") for _ in range(e.nd)]
    torch.cuda.synchronize()
    lo, hi = e.chunks[0]
    sgp = e.ptrs(sg)
    ev = []

    def step(t, timed):
        x = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        x[0].record(stream)
        zero3.zero3_reduce_scatter(e.plan, e.ptrs(e.grads[0]), lo, lo, hi, sgp, zero3.F32, e.sid)
        x[1].record(stream)
        zero3.zero3_adamw_step(e.plan, e.hp, t, sgp, zero3.F32, e.ptrs(e.master), e.ptrs(e.m),
                               e.ptrs(e.v), e.ptrs(e.sparam), lo, hi, e.sid)
        x[2].record(stream)
        zero3.zero3_allgather(e.plan, e.ptrs(e.sparam), e.full.data_ptr(), lo, hi, e.sid)
        x[3].record(stream)
        zero3.zero3_step(e.plan, e.hp, t, e.ptrs(e.grads[0]), lo, e.ptrs(e.master), e.ptrs(e.m),
                         e.ptrs(e.v), e.ptrs(e.sparam), e.full.data_ptr(), None, lo, hi, e.sid)
        x[4].record(stream)
        if timed:
            ev.append(x)

    t = 0
    for _ in range(args.warmup):
        t += 2
        step(t, False)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        t += 2
        step(t, True)
    torch.cuda.synchronize()
    n = hi - lo
    nd = w.n_ranks
    parts = {"reduce_scatter": (0, 1, 2 * nd + 4), "adamw": (1, 2, 4 + 24 + 2),
             "allgather": (2, 3, 2 + 2), "fused": (3, 4, 2 * nd + 28)}
    peak, _ = peaks()
    out = {}
    for k, (i, j, bpe) in parts.items():
        ms = statistics.mean(x[i].elapsed_time(x[j]) for x in ev)
        gbs = n * bpe / (ms / 1e3) / 1e9
        out[k] = {"ms": ms, "bytes_per_elem": bpe, "gbs": gbs, "frac": gbs / peak}
    unf = sum(out[k]["ms"] for k in ("reduce_scatter", "adamw", "allgather"))
    print(json.dumps({"metric": "unfused vs fused ZeRO-3 step (ablation)", "unit": "ms",
                      "config": {"workload": desc, "elements": n},
                      "kernels": out, "unfused_ms": unf, "fused_ms": out["fused"]["ms"],
                      "fusion_speedup": unf / out["fused"]["ms"]}))
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from zero_sharded_optimizer_shard_gb300 import build as b
    if rank == 0 or world == 1:
        b.build_all(quiet=True)
    if world > 1:
        dist.barrier()
    from zero_sharded_optimizer_shard_gb300 import workloads as W, zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation

    fac, state_ranks, bucketed, _ = WORKLOADS[args.workload]
    w = make_workload(args)
    stream = torch.cuda.Stream()
    e = Emulation(w, device=f"cuda:{local}", state_ranks=state_ranks, bucketed=bucketed,
                  stream=stream)
    with torch.cuda.stream(stream):
        e.init_params()
        e.fill_grads(1)   # generated once before timing, reused by every step
    torch.cuda.synchronize()
    nbytes = e.step_bytes()
    n_params = w.psi if state_ranks is None else nbytes["flat_elems"] + e.psi_s

    def full_step(t, ev=None):
        if ev is not None:
            ev[0].record(stream)
        e.forward_backward_gathers()
        if ev is not None:
            ev[1].record(stream)
        for (a_, b_), G in zip(e.chunks, e.grads):
            zero3.zero3_step(e.plan, e.hp, t, e.ptrs(G), a_, e.ptrs(e.master), e.ptrs(e.m),
                             e.ptrs(e.v), e.ptrs(e.sparam), e.full.data_ptr(), None, a_, b_, e.sid)
        if ev is not None:
            ev[2].record(stream)
        zero3.zero3_persistent_step(e.plan, e.hp, t, e.persist, e.sid)
        if ev is not None:
            ev[3].record(stream)

    t = 0
    for _ in range(args.warmup):
        t += 1
        full_step(t)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    tw0 = time.time()
    wall0 = time.perf_counter()
    start.record(stream)
    for k in range(args.steps):
        t += 1
        full_step(t, evs[k])
    end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    tw1 = time.time()
    if world > 1:
        dist.barrier()
    ms = start.elapsed_time(end)
    gather_ms = [x[0].elapsed_time(x[1]) for x in evs]
    fused_ms = [x[1].elapsed_time(x[2]) for x in evs]
    persist_ms = [x[2].elapsed_time(x[3]) for x in evs]
    clk = clocks.stop(tw0, tw1)
    if world > 1:
        ms = reduce_max(ms, f"cuda:{local}")

    # ---- end to end through the public API: host gradients in, params out
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(e, w, args, stream, n_params, t)
        if world > 1 and e2e is not None and e2e.get("ms_per_step"):
            e2e["ms_per_step"] = reduce_max(e2e["ms_per_step"], f"cuda:{local}")
            e2e["value"] = replica_throughput(world, n_params, e2e["ms_per_step"])

    if rank == 0:
        ms_step = ms / args.steps
        fused_launch_ms = statistics.mean(fused_ms) / max(len(e.chunks), 1)
        fused_bytes_launch = nbytes["fused"] / max(len(e.chunks), 1)
        peak, peak_kind = peaks()
        achieved = fused_bytes_launch / (fused_launch_ms / 1e3) / 1e9
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            rate, sample, _ = cpu_oracle_rate(w, budget_s=15.0)
            cpu = {"value": rate, "unit": "params/s", "cores": 1, "kind": "oracle",
                   "sample": sample}
        step_gbs = nbytes["total"] / (ms_step / 1e3) / 1e9
        line = {
            "metric": METRIC,
            "value": replica_throughput(world, n_params, ms_step),
            "unit": "params/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": step_config(args, w, world, e.psi_pad, e.psi_s, nbytes["flat_elems"],
                                  [e.plan.submodule(k)[1]
                                   for k in range(e.plan.info.n_submodules)]),
            "step_gbs": step_gbs,
            "step_hbm_frac": step_gbs / peak,
            "fused_step": {"ms_per_launch": fused_launch_ms, "launches_per_step": len(e.chunks),
                           "bytes_per_launch": fused_bytes_launch,
                           "bytes_per_elem": 2 * w.n_ranks + 28,
                           "params_per_s": nbytes["flat_elems"] / max(len(e.chunks), 1)
                           / (fused_launch_ms / 1e3)},
            # every row of the step, timed by events on the launching stream,
            # against the same measured copy peak as the roofline
            "rows": {
                name: dict(ms_per_step=ms_, launches=n_, bytes=b_,
                           gbs=b_ / ms_ / 1e6 if ms_ > 0 else 0.0,
                           frac=b_ / ms_ / 1e6 / peak if ms_ > 0 else 0.0)
                for name, ms_, n_, b_ in (
                    ("a1_a3_fused", statistics.mean(fused_ms), len(e.chunks), nbytes["fused"]),
                    ("a4_persistent", statistics.mean(persist_ms), 1, nbytes["persistent"]),
                    ("a5_gathers", statistics.mean(gather_ms),
                     launches_per_step(e) - len(e.chunks) - (1 if e.psi_s > 0 else 0),
                     nbytes["gathers"]))
            },
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": profile_traffic(kernels_sha())
                         if (args.workload == "decoder_1p3b" and not args.n_ranks) else None,
                         "kernel": "stream_kernel<kFused, N_d> (zero3_step)"},
            "gpu_launches": launches_per_step(e) * args.steps,
            "clocks": clk,
            "wall_s_timed": wall,
            "cpu_baseline": cpu,
            "e2e": e2e,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(e, w, args, stream, n_params, t0):
    """Same step through the public API with host buffers: every step copies
    every rank's local gradients (and the persistent-group gradients) from
    pinned host memory and reads the full bf16 parameter buffer back into
    pinned host memory.  Pipelined over two device buffer sets: the upload of
    step k+1 and the read-back of step k run on their own streams while step
    k computes; events order every reuse of a buffer."""
    import torch
    from zero_sharded_optimizer_shard_gb300 import zero3
    steps = max(2, min(args.steps, 6))
    need = sum(x.numel() * 2 for G in e.grads for x in G) + e.full.numel() * 2
    free, _ = torch.cuda.mem_get_info()
    if need > free - (2 << 30):
        return {"value": None, "unit": "params/s",
                "note": f"second device buffer set ({need / 1e9:.0f} GB) does not fit"}
    try:
        host_g = [[torch.empty(x.numel(), dtype=x.dtype, pin_memory=True) for x in G] for G in e.grads]
        host_pg = [torch.empty(x.numel(), dtype=x.dtype, pin_memory=True) for x in e.pgrads]
        host_full = torch.empty(e.full.numel(), dtype=e.full.dtype, pin_memory=True)
        dev_g = [e.grads, [[torch.empty_like(x) for x in G] for G in e.grads]]
        dev_pg = [e.pgrads, [torch.empty_like(x) for x in e.pgrads]]
        dev_full = [e.full, torch.empty_like(e.full)]
    except RuntimeError as exc:
        return {"value": None, "unit": "params/s", "error": f"allocation failed: {exc}"}
    for hG, G in zip(host_g, e.grads):
        for h, d in zip(hG, G):
            h.copy_(d)
    for h, d in zip(host_pg, e.pgrads):
        h.copy_(d)
    h2d = sum(x.numel() * 2 for hG in host_g for x in hG) + sum(x.numel() * 2 for x in host_pg)
    d2h = host_full.numel() * 2
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    uploaded = [ev() for _ in range(steps)]
    up_t = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(steps)]
    computed = [ev() for _ in range(steps)]
    read = [ev() for _ in range(steps)]
    torch.cuda.synchronize()
    t = t0
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    start.record(up)
    for k in range(steps):
        b = k % 2
        with torch.cuda.stream(up):
            if k >= 2:
                up.wait_event(computed[k - 2])  # buffer set b was read by step k-2
            up_t[k][0].record(up)
            for hG, G in zip(host_g, dev_g[b]):
                for h, d in zip(hG, G):
                    d.copy_(h, non_blocking=True)
            for h, d in zip(host_pg, dev_pg[b]):
                d.copy_(h, non_blocking=True)
            up_t[k][1].record(up)
            uploaded[k].record(up)
        stream.wait_event(uploaded[k])
        if k >= 2:
            stream.wait_event(read[k - 2])      # full[b] of step k-2 was read back
        t += 1
        e.forward_backward_gathers()
        ps = zero3.persist_state([x.data_ptr() for x in dev_pg[b]], e.pmaster.data_ptr(),
                                 e.pm.data_ptr(), e.pv.data_ptr(), e.pparam.data_ptr())
        for (lo, hi), G in zip(e.chunks, dev_g[b]):
            zero3.zero3_step(e.plan, e.hp, t, e.ptrs(G), lo, e.ptrs(e.master), e.ptrs(e.m),
                             e.ptrs(e.v), e.ptrs(e.sparam), dev_full[b].data_ptr(), None, lo, hi,
                             e.sid)
        zero3.zero3_persistent_step(e.plan, e.hp, t, ps, e.sid)
        computed[k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[k])
            host_full.copy_(dev_full[b], non_blocking=True)
            read[k].record(down)
    end.record(down)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    ms = start.elapsed_time(end) / steps
    up_ms = [a.elapsed_time(b_) for a, b_ in up_t]
    return {"value": n_params / (ms / 1e3), "unit": "params/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms,
            "wall_ms_per_step": wall * 1e3 / steps,
            "upload_ms_per_step": statistics.mean(up_ms),
            "h2d_gbs": h2d / (statistics.mean(up_ms) / 1e3) / 1e9,
            "pipeline": "uploads of step k+1 and read-back of step k overlap step k"}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.stage == 2:
        return run_stage12(args)
    if args.coordinator:
        return run_coordinator(args)
    if args.qwz:
        return run_qwz(args)
    if args.unfused:
        return run_unfused(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
