"""Benchmark of the ZeRO-3 hot path: one step = a forward and a backward
gather of every submodule (bucketed, allgather_bucket_size elements per call)
plus the fused reduce-scatter/AdamW/cast/all-gather step over every virtual
rank and the persistent group.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decoder_1p3b|gpt2_small|ragged|llama_7b_rank0|...]
                    [--second auto|none|<workload>]

Prints one JSON line (rank 0).  The default run measures the 1.3B decoder
(the headline `value`) and, in the same line under `configs`, the Llama-7B
rank-0 view.  N > 1 runs one replica of the workload per GPU (the emulated
ranks live inside each GPU; there is no inter-GPU step), launched by
torch.distributed.run; value is the params of all replicas per second (weak
scaling).  --impl reference times the CPU oracle, as it stands, on the
host's cores on a scaled copy of the same parameter list.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused ZeRO-3 step params/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
PROFILE_JSON = os.path.join(ROOT, "profiles", "zero3_step_fused_decoder_1p3b.json")
# GB300 HBM3e nominal bandwidth (NVIDIA's product figure): the second
# denominator of the roofline, beside the measured copy rate.
NOMINAL_HBM_GBS = 7900.0

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
DEFAULT_SECOND = {"decoder_1p3b": "llama_7b_rank0"}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decoder_1p3b")
    ap.add_argument("--second", default="auto",
                    help="second workload measured in the same run and reported under "
                         "`configs` (auto: the Llama-7B rank-0 view after the 1.3B headline; "
                         "none: skip)")
    ap.add_argument("--n-ranks", type=int, default=None,
                    help="override the workload's N_d (small profiling cases)")
    ap.add_argument("--gather-bucket", type=int, default=None,
                    help="elements per submodule-gather call (allgather_bucket_size; default "
                         "the workload's 5e8; 0 = one call per submodule)")
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
    ap.add_argument("--e2e-copy-streams", type=int, choices=[1, 2], default=2,
                    help="host copies of the end-to-end run on one stream (uploads and "
                         "read-backs in turn) or two (concurrent)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of oracle work per CPU-baseline measurement")
    return ap.parse_args(argv)


def second_workload(args):
    if args.second == "none" or args.n_ranks:
        return None
    if args.second == "auto":
        return DEFAULT_SECOND.get(args.workload)
    if args.second not in WORKLOADS:
        raise SystemExit(f"unknown --second workload {args.second}")
    return args.second if args.second != args.workload else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


FUSED_SOURCES = ("kernels.cu", "device_common.cuh", "internal.h")


def kernels_sha() -> str:
    """Hash of the sources the fused kernel is compiled from (its profile
    figures hold only while these are unchanged)."""
    h = hashlib.sha256()
    for name in FUSED_SOURCES:
        p = os.path.join(ROOT, "zero_sharded_optimizer_shard_gb300", "csrc", name)
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profile_traffic(workload: str, sha: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu
    summary (machine-readable copy), if it was captured on the current
    kernel source; None otherwise."""
    if not os.path.exists(PROFILE_JSON):
        return None
    with open(PROFILE_JSON) as f:
        d = json.load(f)
    if d.get("fused_sources_sha16") != sha:
        return None
    v = d.get("traffic_bytes_per_launch", {}).get(workload)
    return float(v) if v is not None else None


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


def make_workload(args, name=None):
    from zero_sharded_optimizer_shard_gb300 import workloads as W
    name = name or args.workload
    fac = WORKLOADS[name][0]
    w = W.llama_7b(rank0_view=(fac == "llama_7b_rank0")) if fac.startswith("llama_7b") \
        else getattr(W, fac)()
    if getattr(args, "n_ranks", None) and name == args.workload:
        w.n_ranks = args.n_ranks
    if getattr(args, "stage", 3) == 2:
        w.threshold = 0  # the persistence threshold is a stage-3 setting
    gb = getattr(args, "gather_bucket", None)
    if gb is not None:
        w.gather_bucket = gb
    return w


def gather_groups(sub_numels, bucket):
    """Consecutive submodules grouped into all-gather buckets of at most
    `bucket` elements (0: one submodule per group)."""
    groups, cur, size = [], [], 0
    for k, n in enumerate(sub_numels):
        if cur and (bucket <= 0 or size + n > bucket):
            groups.append(cur)
            cur, size = [], 0
        cur.append(k)
        size += n
    if cur:
        groups.append(cur)
    return groups


def step_config(args, w, world, psi_pad, psi_s, n_flat, sub_numels, name=None):
    """The `config` object of the step benchmark, from the partition's sizes
    alone, so that both arms (GPU path and CPU oracle) report the same one.
    Bytes per step: the fused step (2*N_d + 28 per flat element), the
    persistent group (2*N_d + 26) and two gathers of every submodule (4)."""
    name = name or args.workload
    nd = w.n_ranks
    total = n_flat * (2 * nd + 28) + psi_s * (2 * nd + 26) + 2 * sum(sub_numels) * 4
    desc = WORKLOADS[name][3]
    if getattr(args, "n_ranks", None) and name == args.workload:
        desc += f" (N_d overridden to {nd})"
    params = w.psi if WORKLOADS[name][1] is None else n_flat + psi_s
    groups = gather_groups(sub_numels, w.gather_bucket)
    return {
        "workload": desc, "name": name, "n_ranks": nd,
        "params": params, "psi_pad": psi_pad, "psi_s": psi_s,
        "bytes_per_step": total,
        "step": "forward + backward gather of every submodule, fused step with the persistent "
                "group in the same launch",
        "gather_bucket": w.gather_bucket, "gather_calls_per_pass": len(groups),
        "l2": f"inputs larger than L2 ({total / 1e9:.1f} GB touched per step)",
        "grads": "generated once on the device before timing, reused by every step",
        "parallelism": f"{world} replica(s) x {nd} emulated ranks",
    }


# ---------------------------------------------------------------- CPU oracle
def scaled_workload(w, target_params: int):
    """The same parameter list with every tensor scaled by f = target/psi
    (at least one element; zero-size tensors stay empty), the persistence
    threshold moved so that exactly the same tensors stay unpartitioned,
    same N_d, submodules and hyper-parameters.  Returns (workload, f)."""
    import copy
    f = min(1.0, target_params / max(w.psi, 1))
    pers = [n0 > 0 and n0 < w.threshold for n0 in w.numels]
    numels = [0 if n0 == 0 else max(1, int(round(n0 * f))) for n0 in w.numels]
    thr = max([n for n, p in zip(numels, pers) if p] + [0]) + 1
    numels = [n if (p or n0 == 0) else max(n, thr) for n, p, n0 in zip(numels, pers, w.numels)]
    s = copy.copy(w)
    s.numels, s.threshold, s.name = numels, thr, w.name + "_scaled"
    s.bucket = max(1, int(w.bucket * f))
    return s, f


def _oracle_inputs(s, view_rank0: bool):
    """Seeded inputs of the scaled workload (host generator): masters, every
    rank's gradient (rank 0's range only for the rank-0 view), persistent
    group."""
    import numpy as np
    import oracle as O
    from zero_sharded_optimizer_shard_gb300 import synth, workloads as W
    plan = O.partition(s.numels, s.submodule_of, s.n_ranks, s.threshold, s.bucket)
    hi = plan.shard_len if view_rank0 else plan.psi_pad
    mf = np.zeros(plan.psi_pad, np.float32)
    mf[:plan.psi_p] = synth.normal_f32(s.seed, W.STREAM_MASTER, 0, 0, np.arange(plan.psi_p),
                                       s.master_sigma)
    mp = synth.normal_f32(s.seed, W.STREAM_MASTER_PERSIST, 0, 0, np.arange(plan.psi_s),
                          s.master_sigma)
    G = np.zeros((plan.n_ranks, plan.psi_pad), np.uint16)
    n = min(hi, plan.psi_p)
    for q in range(plan.n_ranks):
        G[q, :n] = synth.normal_bf16(s.seed, W.STREAM_GRAD, 1, q, np.arange(n), s.grad_sigma,
                                     s.outlier_p, s.outlier_sigma)
    PG = np.stack([synth.normal_bf16(s.seed, W.STREAM_GRAD_PERSIST, 1, q, np.arange(plan.psi_s),
                                     s.grad_sigma, s.outlier_p, s.outlier_sigma)
                   for q in range(plan.n_ranks)]) if plan.psi_s else \
        np.zeros((plan.n_ranks, 0), np.uint16)
    return dict(mf=mf, mp=mp, G=G, PG=PG, hi=np.int64(hi))


def _oracle_steps(s, inputs, n_steps: int, barrier=None):
    """Runs n_steps whole steps of the oracle, as it stands, on the scaled
    workload: the sharded step over the state ranks' range (reduce-scatter,
    AdamW, bf16 cast, all-gather write), the persistent group, and a forward
    and a backward gather of every submodule.  Returns per-step seconds."""
    import numpy as np
    import oracle as O
    plan = O.partition(s.numels, s.submodule_of, s.n_ranks, s.threshold, s.bucket)
    st, full, ps = O.init_state(plan, inputs["mf"], inputs["mp"])
    G = [inputs["G"][q] for q in range(plan.n_ranks)]
    PG = [inputs["PG"][q] for q in range(plan.n_ranks)]
    hi = int(inputs["hi"])
    order = list(range(plan.n_submodules))
    out = []
    for t in range(1, n_steps + 1):
        if barrier is not None:
            barrier.wait()
        t0 = time.perf_counter()
        for k in order:
            O.fetch_submodule(plan, k, st.sparam, ps.param)
        for k in reversed(order):
            O.fetch_submodule(plan, k, st.sparam, ps.param)
        O.sharded_step(plan, s.hparams, t, G, st, full, 0, hi)
        O.persistent_step(plan, s.hparams, t, PG, ps)
        out.append(time.perf_counter() - t0)
    del np
    return out


def _cpu_worker(s, path, n_steps, barrier, q, wid):
    import numpy as np
    with np.load(path) as z:
        inputs = {k: z[k] for k in z.files}
    q.put((wid, _oracle_steps(s, inputs, n_steps, barrier)))


def oracle_on_cores(s, inputs, n_steps: int, procs: int):
    """The oracle's steps on `procs` host cores at once: procs independent
    copies of the scaled step in spawned processes (one thread each),
    started together at every step.  Returns per-step seconds (the slowest
    process of each step)."""
    import multiprocessing as mp
    import numpy as np
    if procs <= 1:
        return _oracle_steps(s, inputs, n_steps)
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    np.savez(path, **inputs)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    ctx = mp.get_context("spawn")
    barrier, q = ctx.Barrier(procs), ctx.Queue()
    ps = [ctx.Process(target=_cpu_worker, args=(s, path, n_steps, barrier, q, i))
          for i in range(procs)]
    for p in ps:
        p.start()
    res = dict(q.get() for _ in ps)
    for p in ps:
        p.join()
    os.unlink(path)
    return [max(res[i][k] for i in res) for k in range(n_steps)]


def host_mem_available():
    """MemAvailable of /proc/meminfo in bytes, or None where there is none."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def host_cores():
    try:
        aff = len(os.sched_getaffinity(0))
    except AttributeError:
        aff = os.cpu_count() or 1
    return os.cpu_count() or 1, aff


def cpu_oracle_baseline(w, view_rank0: bool, budget_s: float, target_params: int = 2_000_000):
    """The CPU oracle, as it stands, timed on this host's cores: one whole
    step (forward and backward gathers of every submodule, the sharded step
    over the state ranks' range, the persistent group) of the same list
    scaled down to about target_params parameters, single-threaded and on
    every core at once.  params/s = the scaled step's parameters (times the
    processes) / its measured time."""
    s, f = scaled_workload(w, target_params)
    inputs = _oracle_inputs(s, view_rank0)
    import oracle as O
    plan = O.partition(s.numels, s.submodule_of, s.n_ranks, s.threshold, s.bucket)
    params = (plan.shard_len + plan.psi_s) if view_rank0 else s.psi
    one = _oracle_steps(s, inputs, 1)[0]
    n_steps = max(2, min(200, int(budget_s / max(one, 1e-3))))
    single = _oracle_steps(s, inputs, n_steps)
    nproc, aff = host_cores()
    multi = oracle_on_cores(s, inputs, n_steps, aff)
    v1 = params / statistics.mean(single)
    vn = aff * params / statistics.mean(multi)
    return {
        "value": vn, "unit": "params/s", "cores": aff, "kind": "oracle",
        "value_single_thread": v1, "cores_single": 1, "nproc": nproc, "affinity_cores": aff,
        "ms_per_sample_step_single": statistics.mean(single) * 1e3,
        "ms_per_sample_step_all_cores": statistics.mean(multi) * 1e3,
        "sample": (f"the oracle's whole step on the same list scaled by f={f:.3g} "
                   f"({params} params: {len(s.numels)} tensors, same N_d={s.n_ranks}, "
                   f"persistent set and submodules); {n_steps} steps single-threaded, then "
                   f"{aff} processes x {n_steps} steps at once (numpy, one thread each)"),
    }


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle as O
    w = make_workload(args)
    view = WORKLOADS[args.workload][1] is not None
    plan = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    n_flat = plan.shard_len if view else plan.psi_pad
    config = step_config(args, w, args.gpus, plan.psi_pad, plan.psi_s, n_flat,
                         [plan.submodule_numel(k) for k in range(plan.n_submodules)])
    s, f = scaled_workload(w, 2_000_000)
    inputs = _oracle_inputs(s, view)
    sp = O.partition(s.numels, s.submodule_of, s.n_ranks, s.threshold, s.bucket)
    params = (sp.shard_len + sp.psi_s) if view else s.psi
    nproc, aff = host_cores()
    dts = oracle_on_cores(s, inputs, args.warmup + args.steps, aff)[args.warmup:]
    ms = statistics.mean(dts) * 1e3 if dts else float("nan")
    value = aff * params / (ms / 1e3)
    cpu = {"value": value, "unit": "params/s", "cores": aff, "kind": "oracle", "nproc": nproc,
           "sample": (f"the oracle's whole step on the same list scaled by f={f:.3g} "
                      f"({params} params), {aff} processes at once (numpy, one thread each)")}
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # measured: one step of what ran (every core's scaled step)
        "ms_per_step": ms,
        # the oracle's time for one whole step of the full-size workload at
        # the same rate (not timed)
        "extrapolated_ms_per_full_step": config["params"] / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": config,
        "cpu_baseline": cpu,
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


def submodule_pieces(e, k) -> int:
    pieces = 0
    for t, sub in enumerate(e.w.submodule_of):
        if sub != k or e.w.numels[t] == 0:
            continue
        ti = e.plan.tensor(t)
        pieces += 1 if ti.persistent else ti.n_segments
    return pieces


def gather_launches(e, bucket) -> int:
    """Launches of the two gather passes: per zero3_fetch_submodules call
    (one bucket) its pieces in launches of up to 512 (64 when they all fit
    the small description)."""
    n = 0
    for g in gather_groups([e.plan.submodule(k)[1] for k in range(e.plan.info.n_submodules)],
                           bucket):
        p = sum(submodule_pieces(e, k) for k in g)
        n += 2 * (math.ceil(p / 512) if p > 64 else (1 if p > 0 else 0))
    return n


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

    host = {"s": 0.0, "n": 0}

    def one_step(co, t):
        for i, k in enumerate(trace):
            if co is None:
                with torch.cuda.stream(compute):
                    gemms(Wfix, 0, k, i >= n_sub)
                continue
            h0 = time.perf_counter()
            ptr = co.fetch(k)
            host["s"] += time.perf_counter() - h0
            with torch.cuda.stream(compute):
                gemms(arena, (ptr - arena.data_ptr()) // 2, k, i >= n_sub)
            h0 = time.perf_counter()
            co.release(k)
            host["s"] += time.perf_counter() - h0
            host["n"] += 1
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
        host["s"], host["n"] = 0.0, 0
        w0 = time.perf_counter()
        s0.record(compute)
        for _ in range(args.steps):
            t += 1
            one_step(co, t)
        s1.record(compute)
        w1 = time.perf_counter()
        torch.cuda.synchronize()
        results[mode] = {"ms_per_step": s0.elapsed_time(s1) / args.steps,
                         "host_ms_per_step_enqueue": (w1 - w0) * 1e3 / args.steps}
        if host["n"]:
            # host time of one coordinator fetch + release, through the binding
            results[mode]["host_us_per_fetch"] = host["s"] / host["n"] * 1e6
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


def measure(args, name, world, local, with_e2e, with_cpu):
    """The step of workload `name` on this GPU: device-resident timing
    (every row by CUDA events on the launching stream, clocks sampled during
    the timed region), the end-to-end variant through the C ABI with host
    buffers, and the CPU oracle baseline.  Returns the line's fields."""
    import torch
    from zero_sharded_optimizer_shard_gb300 import zero3
    from zero_sharded_optimizer_shard_gb300.emulation import Emulation

    fac, state_ranks, bucketed, _ = WORKLOADS[name]
    w = make_workload(args, name)
    stream = torch.cuda.Stream()
    e = Emulation(w, device=f"cuda:{local}", state_ranks=state_ranks, bucketed=bucketed,
                  stream=stream)
    with torch.cuda.stream(stream):
        e.init_params()
        e.fill_grads(1)   # generated once before timing, reused by every step
    torch.cuda.synchronize()
    nbytes = e.step_bytes()
    n_params = w.psi if state_ranks is None else nbytes["flat_elems"] + e.psi_s
    bucket = w.gather_bucket

    def full_step(t, ev=None):
        if ev is not None:
            ev[0].record(stream)
        e.forward_backward_gathers(bucket=bucket)
        if ev is not None:
            ev[1].record(stream)
        # the persistent group rides in the first chunk's launch
        for c, ((a_, b_), G) in enumerate(zip(e.chunks, e.grads)):
            zero3.zero3_step(e.plan, e.hp, t, e.ptrs(G), a_, e.ptrs(e.master), e.ptrs(e.m),
                             e.ptrs(e.v), e.ptrs(e.sparam), e.full.data_ptr(),
                             e.persist if c == 0 else None, a_, b_, e.sid)
        if ev is not None:
            ev[2].record(stream)

    t = 0
    for _ in range(args.warmup):
        t += 1
        full_step(t)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
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
    ms = start.elapsed_time(end) / args.steps
    gather_ms = [x[0].elapsed_time(x[1]) for x in evs]
    fused_ms = [x[1].elapsed_time(x[2]) for x in evs]
    clk = clocks.stop(tw0, tw1)
    if world > 1:
        ms = reduce_max(ms, f"cuda:{local}")

    e2e = None
    if with_e2e:
        e2e = run_e2e(e, w, args, stream, n_params, t)
        if world > 1 and e2e is not None and e2e.get("ms_per_step"):
            e2e["ms_per_step"] = reduce_max(e2e["ms_per_step"], f"cuda:{local}")
            e2e["value"] = replica_throughput(world, n_params, e2e["ms_per_step"])

    n_fused = max(len(e.chunks), 1)
    fused_bytes = nbytes["fused"] + nbytes["persistent"]
    fused_launch_ms = statistics.mean(fused_ms) / n_fused
    peak, peak_kind = peaks()
    achieved = fused_bytes / n_fused / (fused_launch_ms / 1e3) / 1e9
    n_gather = gather_launches(e, bucket)
    cpu = None
    if with_cpu:
        cpu = cpu_oracle_baseline(w, state_ranks is not None, args.cpu_budget)
    step_gbs = nbytes["total"] / (ms / 1e3) / 1e9
    sha = kernels_sha()
    traffic = None if args.n_ranks else profile_traffic(name, sha)
    res = {
        "value": replica_throughput(world, n_params, ms),
        "unit": "params/s",
        "ms_per_step": ms,
        "config": step_config(args, w, world, e.psi_pad, e.psi_s, nbytes["flat_elems"],
                              [e.plan.submodule(k)[1] for k in range(e.plan.info.n_submodules)],
                              name=name),
        "step_gbs": step_gbs,
        "step_hbm_frac": step_gbs / peak,
        "fused_step": {"ms_per_launch": fused_launch_ms, "launches_per_step": n_fused,
                       "bytes_per_launch": fused_bytes / n_fused,
                       "bytes_per_elem": 2 * w.n_ranks + 28,
                       "gbs": achieved, "frac": achieved / peak,
                       "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                       "params_per_s": (nbytes["flat_elems"] + e.psi_s) / n_fused
                       / (fused_launch_ms / 1e3)},
        # every row of the step, timed by events on the launching stream,
        # against the same measured copy peak as the roofline
        "rows": {
            nm: dict(ms_per_step=ms_, launches=n_, bytes=b_,
                     gbs=b_ / ms_ / 1e6 if ms_ > 0 else 0.0,
                     frac=b_ / ms_ / 1e6 / peak if ms_ > 0 else 0.0)
            for nm, ms_, n_, b_ in (
                ("a1_a4_fused", statistics.mean(fused_ms), n_fused, fused_bytes),
                ("a5_gathers", statistics.mean(gather_ms), n_gather, nbytes["gathers"]))
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "peak_note": "MEASURED_PEAKS.json hbm_gbs: a torch copy, read+write bytes",
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "nominal_note": "GB300 HBM3e nominal bandwidth (NVIDIA product figure)",
                     "traffic": traffic,
                     "traffic_source": (os.path.relpath(PROFILE_JSON, ROOT) + f" (fused kernel "
                                        f"sources {sha})") if traffic is not None else None,
                     "kernel": "stream_kernel<kFused, N_d> (zero3_step)"},
        "gpu_launches": (n_fused + n_gather) * args.steps,
        "clocks": clk,
        "wall_s_timed": wall,
        "cpu_baseline": cpu,
        "e2e": e2e,
    }
    del e
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


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

    head = measure(args, args.workload, world, local, with_e2e=not args.no_e2e,
                   with_cpu=(not args.no_cpu_baseline and world == 1 and rank == 0))
    extra = {}
    second = second_workload(args)
    if second:
        # the host-copy variant of the second workload runs at N = 1 only (its
        # pinned host buffers would be held by every replica at once)
        extra[second] = measure(args, second, world, local,
                                with_e2e=(not args.no_e2e and world == 1),
                                with_cpu=(not args.no_cpu_baseline and world == 1 and rank == 0))
    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": "params/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic"}
        line.update({k: v for k, v in head.items() if k not in line})
        if extra:
            line["configs"] = extra
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(e, w, args, stream, n_params, t0):
    """Same step through the public API with host buffers: every step copies
    every rank's local gradients (and the persistent-group gradients) from
    pinned host memory and reads the parameters the step updated (the state
    ranks' range of the full bf16 buffer) back into pinned host memory.
    Pipelined over two device buffer sets: the upload of step k+1 and the
    read-back of step k run on their own streams while step k computes;
    events order every reuse of a buffer.  Two untimed pipelined steps come
    before the timed ones.  Before the pipelined run, the same copies alone
    measure the host link (one copy per buffer)."""
    import torch
    from zero_sharded_optimizer_shard_gb300 import zero3
    steps = max(2, min(args.steps, 6))
    lo = min(e.state_ranks) * e.S
    hi = min((max(e.state_ranks) + 1) * e.S, e.psi_pad)
    # every rank's gradient buffer per chunk (the first also holds the
    # persistent group's gradients after the flat ones)
    need = sum(x.numel() * 2 for G in e.gbufs for x in G) + e.full.numel() * 2
    free, _ = torch.cuda.mem_get_info()
    if need > free - (2 << 30):
        return {"value": None, "unit": "params/s",
                "note": f"second device buffer set ({need / 1e9:.0f} GB) does not fit"}
    # pinned host memory of every process on this node at once: leave most of
    # the host's available memory alone
    pinned = sum(x.numel() * 2 for G in e.gbufs for x in G) + (hi - lo) * 2
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    avail = host_mem_available()
    if avail is not None and pinned * local_world > 0.6 * avail:
        return {"value": None, "unit": "params/s",
                "note": f"{local_world} x {pinned / 1e9:.0f} GB of pinned host buffers would "
                        f"exceed 60% of the host's {avail / 1e9:.0f} GB available memory"}
    try:
        host_g = [[torch.empty(x.numel(), dtype=x.dtype, pin_memory=True) for x in G]
                  for G in e.gbufs]
        host_full = torch.empty(hi - lo, dtype=e.full.dtype, pin_memory=True)
        dev_g = [e.gbufs, [[torch.empty_like(x) for x in G] for G in e.gbufs]]
        dev_full = [e.full, torch.empty_like(e.full)]
    except RuntimeError as exc:
        return {"value": None, "unit": "params/s", "error": f"allocation failed: {exc}"}
    for hG, G in zip(host_g, e.gbufs):
        for h, d in zip(hG, G):
            h.copy_(d)
    h2d = sum(x.numel() * 2 for hG in host_g for x in hG)
    d2h = host_full.numel() * 2
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    # byte offset of the persistent group's gradients in each rank's first buffer
    poff = e.pgrads[0].data_ptr() - e.gbufs[0][0].data_ptr() if e.gbufs else 0

    def upload(b):
        for hG, G in zip(host_g, dev_g[b]):
            for h, d in zip(hG, G):
                d.copy_(h, non_blocking=True)

    # the host link alone: the same uploads and read-back, nothing else running
    link = {}
    torch.cuda.synchronize()
    for nm, fn, st_, nb in (("h2d", lambda: upload(1), up, h2d),
                            ("d2h", lambda: host_full.copy_(dev_full[1][lo:hi], non_blocking=True),
                             down, d2h)):
        ts = []
        for _ in range(2):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(st_):
                a_.record(st_)
                fn()
                b_.record(st_)
            torch.cuda.synchronize()
            ts.append(a_.elapsed_time(b_))
        link[nm] = nb / (min(ts) / 1e3) / 1e9
    # untimed pipelined steps first: the timed region starts in the steady
    # state, not with the first upload after the link probe's idle gap
    warm = 2
    total = warm + steps
    ev = lambda: torch.cuda.Event()
    uploaded = [ev() for _ in range(total)]
    up_t = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(total)]
    computed = [ev() for _ in range(total)]
    read = [ev() for _ in range(total)]
    # one copy stream: every copy in issue order (upload k+1, then read-back
    # k); two: read-backs on their own stream, concurrent with uploads
    down_s = up if args.e2e_copy_streams == 1 else down

    def enqueue_upload(k):
        with torch.cuda.stream(up):
            if k >= 2:
                up.wait_event(computed[k - 2])  # buffer set k % 2 was read by step k-2
            up_t[k][0].record(up)
            upload(k % 2)
            up_t[k][1].record(up)
            uploaded[k].record(up)

    torch.cuda.synchronize()
    t = t0
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()

    def begin_timing():  # on the upload stream, right before step `warm`'s upload
        nonlocal wall0
        start.record(up)
        wall0 = time.perf_counter()

    if warm == 0:
        begin_timing()
    enqueue_upload(0)
    for k in range(total):
        b = k % 2
        stream.wait_event(uploaded[k])
        if k >= 2:
            stream.wait_event(read[k - 2])      # full[b] of step k-2 was read back
        t += 1
        e.forward_backward_gathers(bucket=w.gather_bucket)
        ps = zero3.persist_state([x.data_ptr() + poff for x in dev_g[b][0]], e.pmaster.data_ptr(),
                                 e.pm.data_ptr(), e.pv.data_ptr(), e.pparam.data_ptr())
        for c, ((clo, chi), G) in enumerate(zip(e.chunks, dev_g[b])):
            zero3.zero3_step(e.plan, e.hp, t, e.ptrs(G), clo, e.ptrs(e.master), e.ptrs(e.m),
                             e.ptrs(e.v), e.ptrs(e.sparam), dev_full[b].data_ptr(),
                             ps if c == 0 else None, clo, chi, e.sid)
        computed[k].record(stream)
        if k + 1 < total:
            if k + 1 == warm:
                begin_timing()
            enqueue_upload(k + 1)               # overlaps step k
        with torch.cuda.stream(down_s):
            down_s.wait_event(computed[k])
            host_full.copy_(dev_full[b][lo:hi], non_blocking=True)
            read[k].record(down_s)
    end.record(down_s)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    ms = start.elapsed_time(end) / steps
    up_t = up_t[warm:]
    up_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in up_t)
    h2d_gbs = h2d / (up_ms / 1e3) / 1e9
    return {"value": n_params / (ms / 1e3), "unit": "params/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "warmup": warm, "ms_per_step": ms,
            "wall_ms_per_step": wall * 1e3 / steps,
            "upload_ms_per_step": up_ms,
            "upload_ms_each": [round(a.elapsed_time(b_), 3) for a, b_ in up_t],
            "h2d_gbs": h2d_gbs,
            "h2d_link_gbs": link["h2d"], "d2h_link_gbs": link["d2h"],
            "h2d_frac": h2d_gbs / link["h2d"],
            "bound_ms_per_step": max(h2d / link["h2d"], d2h / link["d2h"]) / 1e6,
            "link_note": "host link measured in the same run: the same pinned buffers copied "
                         "alone, one copy per buffer, best of 2",
            "copy_streams": args.e2e_copy_streams,
            "pipeline": ("upload of step k+1 overlaps step k; read-back of step k follows it on "
                         "the same copy stream" if args.e2e_copy_streams == 1 else
                         "upload of step k+1 and read-back of step k overlap step k, on two "
                         "copy streams")}


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
