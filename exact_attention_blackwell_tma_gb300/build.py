"""Build libattn.so (and the GPU self-test library) in-tree with nvcc for sm_103a.

Each .cu file is compiled separately (in parallel) and linked into a shared
library next to this file. A library is rebuilt when any of its sources or the
headers it may include is newer than it. No cmake, no torch extension build.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")

LIBS = {
    "libattn.so": ["api.cu", "fwd.cu", "fwd_wide.cu", "bwd.cu", "bwd_wide.cu", "bwd_pair.cu"],
    "libattn_selftest.so": ["selftest.cu"],
}
HEADERS = ["ptx.cuh", "sched.cuh", "kernels.h", "mask.cuh", "dq_order.cuh", "dq_reduce.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def lib_path(name: str = "libattn.so") -> str:
    return os.path.join(PKG, name)


def _flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                   "--expt-relaxed-constexpr", *extra]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, verbose: bool, extra=()) -> str:
    cmd = [nvcc(), *_flags(extra), "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return res.stderr


def build(verbose: bool = False, force: bool = False, jobs: int | None = None) -> list:
    """Compile every library; returns the paths of the built shared objects."""
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "attn.h")]
    tasks = []
    for lib, srcs in LIBS.items():
        for s in srcs:
            src = os.path.join(CSRC, s)
            obj = os.path.join(BUILD, s.replace(".cu", ".o"))
            if force or _stale(obj, [src] + headers):
                tasks.append((src, obj))
    logs = []
    if tasks:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(tasks), os.cpu_count() or 4)) as ex:
            futs = [ex.submit(_compile, s, o, verbose) for s, o in tasks]
            for f in futs:
                logs.append(f.result())
    out = []
    for lib, srcs in LIBS.items():
        objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in srcs]
        target = lib_path(lib)
        if force or _stale(target, objs):
            tmp = target + f".tmp{os.getpid()}"
            cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"link of {lib} failed:\n{res.stdout}\n{res.stderr}")
            os.replace(tmp, target)
        out.append(target)
    if verbose:
        for l in logs:
            sys.stderr.write(l)
    return out


if __name__ == "__main__":
    for p in build(verbose="-v" in sys.argv, force="-f" in sys.argv):
        print(p)
