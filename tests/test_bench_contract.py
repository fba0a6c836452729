"""The benchmark's one-line JSON contract: the reference arm (CPU oracle)
runs here; our arm runs on the GPU with a small workload."""
import json
import os
import subprocess
import sys

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
    d = run_bench("--impl", "reference", "--workload", "gpt2_small", "--steps", "1",
                  "--warmup", "0")
    assert BASE_KEYS <= set(d) and d["impl"] == "reference"
    assert d["unit"] == "params/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] and d["config"]["bytes_per_step"] > 0
    assert d["ms_per_step"] > 0


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
    assert set(rows) == {"a1_a3_fused", "a4_persistent", "a5_gathers"}
    assert all(0 < r["frac"] < 2 and r["launches"] >= 1 for r in rows.values())
    assert rows["a1_a3_fused"]["frac"] == pytest.approx(r["frac"], rel=1e-6)
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
