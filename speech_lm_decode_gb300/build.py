"""Builds libq3tts.so (sm_103a) in-tree with nvcc: one object per .cu, in parallel."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libq3tts.so")
SOURCES = ["linear.cu", "gemm_tc.cu", "attention.cu", "sampler.cu", "loop.cu", "persist.cu", "cluster_step.cu", "q3tts.cu",
           "noalloc.cu", "codec.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers += [os.path.join(ROOT, "include", f) for f in ("q3tts.h", "q3codec.h")]
    procs, objs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            cmd = [nvcc()] + ARCH + FLAGS + ["-c", s, "-o", o]
            if verbose:
                cmd.append("-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(failed))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"])
        os.replace(tmp, LIB)
    return LIB


def build_calibration() -> str:
    """The GEMM shape calibration tool (calibrate_gemm.cu; not part of the
    library): gemm_tc.cu and linear.cu compiled with Q3_GEMM_CALIBRATION."""
    os.makedirs(BUILD, exist_ok=True)
    out = os.path.join(BUILD, "calibrate_gemm")
    srcs = [os.path.join(HERE, "calibrate_gemm.cu"), os.path.join(CSRC, "gemm_tc.cu"), os.path.join(CSRC, "linear.cu")]
    subprocess.check_call([nvcc()] + ARCH + FLAGS + ["-DQ3_GEMM_CALIBRATION", "-o", out] + srcs + ["-lcuda"])
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
