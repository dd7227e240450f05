"""Build libmt.so in-tree: nvcc for the sm_103a kernels, g++ for the host runtime.

Run ``python -m host_memory_streamed_gb300.build`` (or ``__graft_entry__.build()``).
Objects go to ``_build/`` next to this file; the library to ``libmt.so``.
Compiles only what changed (by modification time, headers included) and runs
the compilers in parallel.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmt.so")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                     f"-I{INCLUDE}", f"-I{CSRC}"] + os.environ.get("MT_NVCC_EXTRA", "").split()
CXX_FLAGS = ["-O3", "-fPIC", "-std=c++17", "-pthread", "-fno-fast-math", "-fno-math-errno", "-Wall", "-Wno-unused-function",
             f"-I{INCLUDE}", f"-I{CSRC}", f"-I{os.path.join(CUDA_HOME, 'include')}"]


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(src, obj, hdr_mtime):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or hdr_mtime > t


def _compile(src, obj, verbose):
    if src.endswith(".cu"):
        cmd = [NVCC] + NVCC_FLAGS + ["-c", src, "-o", obj]
        if verbose:
            cmd[1:1] = ["-Xptxas", "-v"]
    else:
        cmd = [os.environ.get("CXX", "g++")] + CXX_FLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return (src, r.stderr if verbose else "")


def build(verbose: bool = False, jobs: int | None = None) -> str:
    """Compile every source under csrc/ and link libmt.so; returns its path."""
    if not os.path.exists(NVCC):
        raise RuntimeError(f"nvcc not found at {NVCC}")
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    hdr_mtime = max([os.path.getmtime(h) for h in _headers()] + [0.0])
    stamp = os.path.join(BUILD, "flags.txt")
    flags = " ".join(NVCC_FLAGS + CXX_FLAGS)
    if not os.path.exists(stamp) or open(stamp).read() != flags:
        verbose_all = True
        with open(stamp, "w") as f:
            f.write(flags)
    else:
        verbose_all = False
    objs, todo = [], []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s) + ".o")
        objs.append(o)
        if verbose or verbose_all or _stale(s, o, hdr_mtime):
            todo.append((s, o))
    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for src, log in ex.map(lambda so: _compile(so[0], so[1], verbose), todo):
                if verbose and log:
                    print(f"== {os.path.basename(src)}\n{log}", file=sys.stderr)
    lib_mtime = os.path.getmtime(LIB) if os.path.exists(LIB) else -1
    if todo or lib_mtime < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        shutil.move(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
