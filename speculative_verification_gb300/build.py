"""Compile libss.so (the sm_103a CUDA kernels + C ABI) in-tree with nvcc.

Three translation units compiled in parallel, one -gencode (sm_103a), no cmake; the output goes to
speculative_verification_gb300/_build/libss.so.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libss.so")
SOURCES = ["ss_kernel.cu", "ss_hist.cu", "ss_shard.cu", "ss_fused.cu"]
DEPS = ["ss_kernel.cu", "ss_hist.cu", "ss_hist.h", "ss_shard.cu", "ss_fused.cu", "ss_philox.cuh", "ss_ptx.cuh", "ss_nvtx.h"]

NVCC_FLAGS = [
    "-std=c++17", "-O3", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC",
]
LINK_FLAGS = ["-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-ldl"]


def nvcc():
    cand = os.environ.get("NVCC") or os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    inputs = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(INCLUDE, "ss.h")]
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(map(os.path.getmtime, inputs)):
        return LIB
    # one object per translation unit, compiled in parallel, then one link
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc()] + NVCC_FLAGS + ["-I" + INCLUDE, "-c", "-o", obj, os.path.join(CSRC, src)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd)))
        objs.append(obj)
    failed = [src for src, p in procs if p.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, "nvcc " + " ".join(failed))
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.check_call([nvcc()] + LINK_FLAGS + ["-o", tmp] + objs)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
