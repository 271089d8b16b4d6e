"""Build the decoder's C-ABI shared library for sm_103a (in-tree).

    python -m ctc_prefix_beam_gb300.build

compiles ``csrc/*.cu`` in parallel with nvcc and links
``ctc_prefix_beam_gb300/_build/libctcpb.so`` (CUDA runtime linked statically,
so the library only needs the driver at run time).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libctcpb.so")
SOURCES = ["ctcpb_kernels.cu", "ctcpb_warp.cu", "ctcpb_rank.cu", "ctcpb_api.cu", "ctcpb_noalloc.cu",
           "ctcpb_selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: no implicit multiply-add contraction anywhere (the decoder's
# float arithmetic is written with explicit round-to-nearest intrinsics).
# CTCPB_PHASE_PROF=1 in the environment builds the per-phase cycle counters.
EXTRA = ["-DCTCPB_PHASE_PROF"] if os.environ.get("CTCPB_PHASE_PROF") == "1" else []
FLAGS = EXTRA + ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the decoder")


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths += [os.path.join(ROOT, "include", "ctcpb.h"), os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "flags.txt")
    flags = " ".join(EXTRA)
    same_flags = os.path.exists(stamp) and open(stamp).read() == flags
    if not force and same_flags and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    with open(stamp, "w") as f:
        f.write(flags)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        with open(os.path.join(BUILD, src + ".log"), "w") as f:
            f.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{p.stderr[-4000:]}")
        if verbose:
            sys.stderr.write(p.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stderr[-4000:]}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
