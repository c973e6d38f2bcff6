"""Build the in-tree shared library libfa_gb300.so with nvcc (sm_103a only).

Usage: ``python -m tiled_attention_fwd_gb300.build [--force] [--verbose]``.
Translation units compile in parallel; object files go to ``_build/`` next to
this file and the library to this package directory.  The build is skipped
when the library is newer than every source file.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import glob
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa_gb300.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"] + ARCH_FLAGS


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit's bin/ on PATH")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    stamp = os.path.join(BUILD, "host.txt")
    if not os.path.exists(stamp) or open(stamp).read().strip() != platform.machine():
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every CUDA source and link the library; returns its path."""
    if not force and not ptxas_info and up_to_date():
        return LIB
    nvcc = nvcc_path()
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    objs, logs = [], []
    workers = min(len(sources()), os.cpu_count() or 4)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for src, obj, r in ex.map(compile_one, sources()):
            logs.append((src, r.stdout + r.stderr))
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            objs.append(obj)
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, "-shared", *ARCH_FLAGS, "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(os.path.join(BUILD, "host.txt"), "w") as f:
        f.write(platform.machine())
    if verbose or ptxas_info:
        for src, log in logs:
            if log.strip():
                print(f"== {os.path.basename(src)}\n{log}", file=sys.stderr)
    return LIB


def ptxas_report(names=None):
    """Compile translation units with -Xptxas -v (objects discarded) and return
    {kernel_name: {"registers": int, "spill_stores": int, "spill_loads": int}}."""
    import re
    import tempfile

    nvcc = nvcc_path()
    srcs = [s for s in sources() if names is None or os.path.basename(s) in names]
    out = {}

    def one(src):
        with tempfile.TemporaryDirectory() as td:
            cmd = [nvcc, *NVCC_FLAGS, "-Xptxas", "-v", "-I", INCLUDE, "-c", src, "-o", os.path.join(td, "x.o")]
            return subprocess.run(cmd, capture_output=True, text=True)

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs) or 1) as ex:
        for r in ex.map(one, srcs):
            if r.returncode != 0:
                raise RuntimeError(r.stderr)
            cur = None
            for line in r.stderr.splitlines():
                m = re.search(r"Compiling entry function '([^']+)'", line)
                if m:
                    cur = m.group(1)
                    out[cur] = {}
                m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
                if m and cur:
                    out[cur]["spill_stores"] = int(m.group(1))
                    out[cur]["spill_loads"] = int(m.group(2))
                m = re.search(r"Used (\d+) registers", line)
                if m and cur:
                    out[cur]["registers"] = int(m.group(1))
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / spills / shared memory")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info))


if __name__ == "__main__":
    main()
