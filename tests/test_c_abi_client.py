"""The C ABI from a plain C99 program: tests/c_abi_client.c includes
include/zero3.h with warnings as errors and -pedantic, links libzero3.so and
calls the host-side entry points (planner, placement, accounting, status
text) with the pages' worked examples.  No GPU needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_client(lib, tmp_path):
    from zero_sharded_optimizer_shard_gb300 import build
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(build.lib_path("libzero3.so"))
    exe = str(tmp_path / "c_abi_client")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi_client.c"), "-o", exe,
                        "-L", libdir, "-lzero3", f"-Wl,-rpath,{libdir}", "-lm"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


@pytest.mark.gpu
def test_c_client_runs_the_fused_step(lib, tmp_path):
    """tests/c_abi_step.c allocates every buffer with the CUDA runtime, runs
    three fused steps with the persistent group through the C ABI and writes
    the results; they equal the oracle's three steps on the same inputs
    (rebuilt here from the program's formulas), bit for bit.  Three ranks:
    S = 2667, so two of the ranks' shards sit at nonzero phases in `full`."""
    import numpy as np
    import oracle as O
    from zero_sharded_optimizer_shard_gb300 import build
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.fail("no C compiler on the GPU machine")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cudalib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.exists(os.path.join(d, "libcudart.so"))), None)
    assert cudalib, "libcudart.so not found under CUDA_HOME"
    libdir = os.path.dirname(build.lib_path("libzero3.so"))
    exe, out = str(tmp_path / "c_abi_step"), str(tmp_path / "step.bin")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-ffp-contract=off", "-I", os.path.join(ROOT, "include"),
                        "-isystem", os.path.join(cuda, "include"),
                        os.path.join(ROOT, "tests", "c_abi_step.c"), "-o", exe,
                        "-L", libdir, "-lzero3", "-L", cudalib, "-lcudart",
                        f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe, out], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr

    numels, nr = [3000, 10, 5000, 37], 3
    plan = O.partition(numels, None, nr, 100, 500_000_000)
    S, P, PP, PS = plan.shard_len, plan.psi_pad, plan.psi_p, plan.psi_s
    assert (S, P, PS) == (2667, 8001, 47)
    f32 = np.float32
    f = np.arange(P, dtype=np.int64)
    j = np.arange(PS, dtype=np.int64)
    mf = np.where(f < PP, ((f % 2001) - 1000).astype(f32) / f32(1024), f32(0)).astype(f32)
    mp = (((j % 301) - 150).astype(f32) / f32(512)).astype(f32)

    def bf16(x):  # exact: every value holds at most 8 significant bits
        return (np.asarray(x, f32).view(np.uint32) >> 16).astype(np.uint16)

    G = [np.where(f < PP, bf16((((3 * f + 5 * q) % 41) - 20).astype(f32) / f32(256)), 0)
         .astype(np.uint16) for q in range(nr)]
    PG = [bf16((((7 * j + 3 * q) % 29) - 14).astype(f32) / f32(128)) for q in range(nr)]
    hp = dict(lr=5e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    st, full, ps = O.init_state(plan, mf, mp)
    for t in (1, 2, 3):
        O.sharded_step(plan, hp, t, G, st, full)
        O.persistent_step(plan, hp, t, PG, ps)

    raw = open(out, "rb").read()
    pos = 0

    def take(n, dt):
        nonlocal pos
        a = np.frombuffer(raw, dt, n, pos)
        pos += n * np.dtype(dt).itemsize
        return a

    for q in range(nr):
        assert np.array_equal(take(S, np.uint32), st.master[q].view(np.uint32)), f"master {q}"
    assert np.array_equal(take(P, np.uint16), full), "full"
    assert np.array_equal(take(PS, np.uint32), ps.master.view(np.uint32)), "persistent master"
    assert np.array_equal(take(PS, np.uint16), ps.param), "persistent param"
    assert pos == len(raw)
