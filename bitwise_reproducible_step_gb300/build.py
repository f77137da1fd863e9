"""Build librepstep.so (the CUDA kernels and the C ABI of include/repstep.h) in-tree.

nvcc for sm_103a only, with explicit rounding kept by -fmad=false on device code and
-ffp-contract=off on host code.  Translation units compile in parallel; the shared
library links the CUDA runtime statically so it does not depend on which libcudart the
calling process loaded.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "librepstep.so")
SOURCES = ["repstep.cu", "k_reduce.cu", "k_reduce_ftz.cu", "k_adamw.cu", "k_adamw_ftz.cu",
           "k_small.cu", "k_blake2b.cu", "noalloc.cu", "k_fused.cu", "k_fused_ftz.cu",
           "k_fused_wide.cu", "k_fused_wide_ftz.cu"]
HEADERS = ["common.cuh", "kernels.h", "k_reduce.cuh", "k_adamw.cuh", "merkle.h",
           "adamw_math.cuh", "k_fused.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xptxas=-v",
    "-Xcompiler", "-fPIC,-ffp-contract=off,-fno-fast-math",
    "-I", os.path.join(ROOT, "include"),
]


def _nvcc():
    for cand in [shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]:
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librepstep.so")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "repstep.h")]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append([nvcc, *NVCC_FLAGS, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, r in ex.map(run, jobs):
                if r.returncode != 0 or verbose:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
