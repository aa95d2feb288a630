"""The boundary from C: the header compiles as strict C99 and a C program
linked against the library drives its host-only entry points (plan, work
order, error reporting) without a GPU."""
import os
import shutil
import subprocess

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_dir():
    __graft_entry__.build()
    return os.path.join(ROOT, "attention_forward_sm100_gb300")


def test_c_caller_plans_and_schedules(lib_dir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "plan_example")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "plan_example.c"), "-L", lib_dir, "-lattn_fwd",
           "-Wl,-rpath," + lib_dir, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"


@pytest.mark.gpu
def test_c_program_runs_forward_on_gpu(lib_dir, tmp_path):
    """A C program (CUDA runtime for device memory, the library for
    everything else) runs a causal forward with Q = 0, whose result has a
    closed form: O_i = mean of V_0..V_i, LSE_i = ln(i + 1)."""
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if cc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("no C compiler or CUDA headers")
    exe = str(tmp_path / "run_example")
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(d)]
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "run_example.c"), "-L", lib_dir,
           "-lattn_fwd", "-Wl,-rpath," + lib_dir]
    for d in libdirs:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-lcudart", "-lm", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")


@pytest.mark.gpu
def test_c_host_cost(lib_dir, tmp_path):
    """A C caller's host time per attn_fwd call on the 128-token workload
    shape (the number is printed; the bound only catches a gross
    regression such as re-encoding every tensor map through a slow path)."""
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if cc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("no C compiler or CUDA headers")
    exe = str(tmp_path / "host_cost")
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(d)]
    cmd = [cc, "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "host_cost.c"), "-L", lib_dir,
           "-lattn_fwd", "-Wl,-rpath," + lib_dir]
    for d in libdirs:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-lcudart", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    fields = r.stdout.split()
    assert fields[-1] == "ok"
    enqueue_us = float(fields[fields.index("enqueue_us") + 1])
    assert enqueue_us < 50.0
