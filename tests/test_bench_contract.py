"""The benchmark's one-line JSON contract: the reference arm (CPU oracle)
runs here; our arm runs on the GPU with a small workload."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
             "cpu_baseline", "e2e"}


def run_bench(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    t0 = time.time()
    d = run_bench("--impl", "reference", "--workload", "gpt2_small", "--steps", "2",
                  "--warmup", "1")
    wall = time.time() - t0
    assert BASE_KEYS <= set(d) and d["impl"] == "reference"
    assert d["unit"] == "params/s" and d["value"] > 0 and d["higher_is_better"] is True
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["nproc"] >= cpu["cores"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] and d["config"]["bytes_per_step"] > 0
    # ms_per_step is what was timed: the timed steps fit in the run's own wall clock
    assert 0 < d["ms_per_step"] and d["steps"] * d["ms_per_step"] / 1e3 < wall
    assert d["extrapolated_ms_per_full_step"] > d["ms_per_step"]


def test_scaled_oracle_sample_keeps_the_partition_shape():
    """The CPU baseline's sample is the same list scaled down: same tensor
    count, same persistent set, same submodules and N_d."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle as O
    from zero_sharded_optimizer_shard_gb300 import workloads as W
    for w in (W.decoder_1p3b(), W.llama_7b(), W.ragged(), W.gpt2_small()):
        s, f = bench.scaled_workload(w, 2_000_000)
        assert 0 < f < 1 and len(s.numels) == len(w.numels)
        assert abs(s.psi - 2_000_000) / 2_000_000 < 0.2
        a = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
        b = O.partition(s.numels, s.submodule_of, s.n_ranks, s.threshold, s.bucket)
        assert a.persistent == b.persistent and a.n_submodules == b.n_submodules
        assert [x == 0 for x in w.numels] == [x == 0 for x in s.numels]


@pytest.mark.gpu
def test_our_arm_line():
    d = run_bench("--workload", "gpt2_small", "--steps", "3", "--warmup", "3")
    assert BASE_KEYS <= set(d) and d["n_gpus"] == 1 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["dtype"] == "f32"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 2
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0 and {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    rows = d["rows"]
    assert set(rows) == {"a1_a4_fused", "a5_gathers"}
    assert all(0 < x["frac"] < 2 and x["launches"] >= 1 for x in rows.values())
    assert rows["a1_a4_fused"]["frac"] == pytest.approx(r["frac"], rel=1e-6)
    assert rows["a1_a4_fused"]["launches"] == 1  # persistent group in the same launch
    assert 0 < r["frac_of_nominal"] < r["frac"]
    cpu = d["cpu_baseline"]
    assert cpu["value_single_thread"] > 0 and cpu["nproc"] >= cpu["cores"] >= 1
    assert e["h2d_link_gbs"] > 0 and e["d2h_link_gbs"] > 0 and 0 < e["h2d_frac"] < 1.5
    assert "configs" not in d  # no second workload after gpt2_small by default
    # the reference arm reports the same workload description
    ref = run_bench("--impl", "reference", "--workload", "gpt2_small", "--steps", "1",
                    "--warmup", "0")
    assert ref["config"] == d["config"]
    assert (ref["metric"], ref["unit"], ref["higher_is_better"]) == \
        (d["metric"], d["unit"], d["higher_is_better"])


@pytest.mark.parametrize("workload", ["gpt2_small", "ragged", "decoder_1p3b", "llama_7b_full",
                                      "llama_7b_rank0"])
def test_arms_describe_the_same_workload(workload, lib):
    """The GPU arm builds its config from the C library's plan, the reference
    arm from the oracle's partition: for every workload they must agree (the
    planner runs on the host, so no GPU is needed)."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    import oracle as O
    from zero_sharded_optimizer_shard_gb300 import zero3
    if workload not in bench.WORKLOADS:
        pytest.skip(f"no bench workload {workload}")
    args = argparse.Namespace(workload=workload, n_ranks=None, stage=3)
    w = bench.make_workload(args)
    view = bench.WORKLOADS[workload][1] is not None
    p = O.partition(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    ref = bench.step_config(args, w, 1, p.psi_pad, p.psi_s, p.shard_len if view else p.psi_pad,
                            [p.submodule_numel(k) for k in range(p.n_submodules)])
    plan = zero3.Plan(w.numels, w.submodule_of, w.n_ranks, w.threshold, w.bucket)
    info = plan.info
    ours = bench.step_config(args, w, 1, info.psi_pad, info.psi_s,
                             info.shard_len if view else info.psi_pad,
                             [plan.submodule(k)[1] for k in range(info.n_submodules)])
    assert ours == ref


@pytest.mark.gpu
def test_second_workload_in_the_same_line():
    """A second workload is measured in the same run and reported under
    `configs` with its own roofline, rows, CPU baseline and e2e."""
    d = run_bench("--workload", "gpt2_small", "--second", "ragged", "--steps", "3",
                  "--warmup", "3", "--cpu-budget", "1")
    c = d["configs"]["ragged"]
    assert c["config"]["name"] == "ragged" and c["value"] > 0
    assert 0 < c["roofline"]["frac"] < 2 and c["cpu_baseline"]["value"] > 0
    assert c["e2e"]["value"] > 0 and set(c["rows"]) == {"a1_a4_fused", "a5_gathers"}


def test_fused_profile_matches_the_current_sources():
    """The committed ncu traffic figure belongs to the fused kernel as it is
    now: its JSON is keyed by the hash of the kernel's sources, and the
    bench reads it (for both workloads of the default run) only on a match."""
    sys.path.insert(0, ROOT)
    import bench
    d = json.load(open(bench.PROFILE_JSON))
    assert d["fused_sources_sha16"] == bench.kernels_sha()
    for name in ("decoder_1p3b", "llama_7b_rank0"):
        t = bench.profile_traffic(name, bench.kernels_sha())
        assert t is not None and t > 0
    # within a few per cent of the algorithmic bytes of one launch
    alg_1p3b = 1_315_080_192 * 44 + 643_072 * 42
    assert 0.95 < bench.profile_traffic("decoder_1p3b", bench.kernels_sha()) / alg_1p3b < 1.02
    assert bench.profile_traffic("decoder_1p3b", "0" * 16) is None


@pytest.mark.gpu
@pytest.mark.parametrize("mode", [
    ("--qwz",), ("--qwz", "--qwz-bits", "4"), ("--stage", "2"), ("--unfused",),
    ("--coordinator", "--tokens", "256"), ("--workload", "ragged", "--no-e2e", "--no-cpu-baseline"),
])
def test_other_modes_print_a_line(mode):
    """The bench's other measurement modes on the GPT-2-small list (the
    ragged list for its own mode): each exits 0 and prints one JSON line with
    positive timings."""
    args = list(mode)
    if "--workload" not in args:
        args += ["--workload", "gpt2_small"]
    d = run_bench(*args, "--steps", "2", "--warmup", "1")
    if "--qwz" in mode:
        assert d["fused_qwz"]["gbs"] > 0 and d["allgather_qwz"]["gbs"] > 0
        assert d["config"]["workload"].endswith(f"qwZ int{mode[-1] if len(mode) > 1 else 8} "
                                                "all-gather (block 256)")
    elif "--unfused" in mode:
        assert all(d["kernels"][k]["ms"] > 0 for k in ("reduce_scatter", "adamw", "allgather",
                                                       "fused"))
    elif "--coordinator" in mode:
        assert set(d["modes"]) == {"prefetch", "on_demand", "gemm_only"}
        assert d["modes"]["prefetch"]["stats"]["prefetched"] > 0
    else:
        assert d["value"] > 0 and d["ms_per_step"] > 0
