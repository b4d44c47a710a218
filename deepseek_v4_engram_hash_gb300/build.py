"""Build libengram.so and libengram_synth.so in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel (`nvcc -c`), then one `nvcc -shared`
links the library.  A library is rebuilt only when a source or header is newer
than it.  No cmake, no torch extension machinery.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]

ENGRAM_SRCS = ["api.cu", "hash.cu", "rows.cu", "gemv.cu", "gemm.cu", "gemm_simt.cu", "gemm_tc.cu", "gemm_tc2.cu",
               "gate.cu", "noalloc.cu", "selftest.cu"]
SYNTH_SRCS = ["synth.cu"]

LIBENGRAM = os.path.join(PKG, "libengram.so")
LIBSYNTH = os.path.join(PKG, "libengram_synth.so")


def _newest_input(srcs) -> float:
    deps = [os.path.join(CSRC, s) for s in srcs]
    deps += glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return max(os.path.getmtime(p) for p in deps)


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC] + FLAGS + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def _link(objs, out: str, libs=()):
    tmp = out + f".{os.getpid()}.tmp"
    cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + list(objs) + list(libs)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed for {out}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> None:
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    for out, srcs in ((LIBENGRAM, ENGRAM_SRCS), (LIBSYNTH, SYNTH_SRCS)):
        if force or not os.path.exists(out) or os.path.getmtime(out) < _newest_input(srcs):
            jobs.append((out, srcs))
    if not jobs:
        return
    with cf.ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        futs = {out: [ex.submit(_compile, s, extra_flags) for s in srcs] for out, srcs in jobs}
        for out, fl in futs.items():
            objs = [f.result() for f in fl]
            _link(objs, out)
            if verbose:
                print("built", out)


if __name__ == "__main__":
    build(force=True, verbose=True)
