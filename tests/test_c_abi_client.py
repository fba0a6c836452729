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
