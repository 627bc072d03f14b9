"""Compile the C oracle into oracle/_build/liboracle.so (test infrastructure).

Plain gcc, no fast-math and no FMA contraction, so every fp32 step of the
oracle is one IEEE single rounding on both x86-64 and aarch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rq_oracle.c")
HDR = os.path.join(HERE, "rq_oracle.h")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its sources."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        lib_t = os.path.getmtime(LIB)
        if lib_t >= max(os.path.getmtime(SRC), os.path.getmtime(HDR)):
            return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
