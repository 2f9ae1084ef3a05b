"""Compile the CPU oracle (plain C) into oracle/_build/liboracle.so.

Test infrastructure only.  Building the checker is not using it: the package's
build step compiles it next to the CUDA library so that the tests, the smoke
check and the benchmark's CPU-baseline leg find it on any machine.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ss_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= max(
        os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "ss_oracle.h"))
    ):
        return OUT
    cc = os.environ.get("CC", "cc")
    tmp = OUT + ".tmp%d" % os.getpid()
    cmd = [cc, "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force=True))
