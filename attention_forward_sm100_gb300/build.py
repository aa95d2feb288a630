"""Builds libattn_fwd.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel into _build/ and
linked into attention_forward_sm100_gb300/libattn_fwd.so (CUDA runtime linked
statically, driver entry points resolved at run time). The ptxas report of
each persistent kernel is checked: it must be allocated exactly 128 registers
per thread (the kernel redistributes them between warpgroups with setmaxnreg,
whose budget is computed from that number) and may spill at most a few words.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import platform
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build", platform.machine())
LIB_PATH = os.path.join(HERE, "libattn_fwd.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                 "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]
PERSISTENT_KERNELS = ("fa_tc05_kernel",)
REGS_EXPECTED = 128
SPILL_LIMIT = 64   # bytes of local-memory spill tolerated per persistent kernel


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; set NVCC")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps_mtime():
    files = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def _check_ptxas(log: str, src: str):
    """Checks register allocation and spills of the persistent kernels."""
    entries = re.split(r"ptxas info\s*: Compiling entry function", log)
    for chunk in entries[1:]:
        name = chunk.split("'")[1] if "'" in chunk else ""
        if not any(k in name for k in PERSISTENT_KERNELS):
            continue
        m = re.search(r"Used (\d+) registers", chunk)
        spills = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", chunk)
        if m is None:
            raise RuntimeError(f"{src}: no register report for {name}")
        if int(m.group(1)) != REGS_EXPECTED:
            raise RuntimeError(f"{src}: {name} uses {m.group(1)} registers, the register split needs "
                               f"exactly {REGS_EXPECTED}")
        if spills and max(int(spills.group(1)), int(spills.group(2))) > SPILL_LIMIT:
            raise RuntimeError(f"{src}: {name} spills ({spills.group(0)})")
        if spills and int(spills.group(1)):
            print(f"warning: {src}: {name}: {spills.group(0)}", file=sys.stderr)


def _compile(src: str, force: bool) -> str:
    obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
    log_path = obj + ".ptxas.txt"
    if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _deps_mtime()):
        return obj
    cmd = [_nvcc()] + CFLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log_path, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr[-6000:]}")
    _check_ptxas(r.stdout + r.stderr, os.path.basename(src))
    return obj


def build(force: bool = False, jobs: int | None = None) -> str:
    """Compiles (incrementally) and links the library; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = _sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with concurrent.futures.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, force), srcs))
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB_PATH + ".tmp"
        cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
