"""Compile the CPU oracle (test infrastructure) into oracle/liboracle_adaln.so.

Plain g++, fp64, no fast-math and no FMA contraction, so that the oracle gives
the same bits on x86-64 and aarch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "adaln_oracle.cpp")
HDR = os.path.join(HERE, "adaln_oracle.h")
LIB = os.path.join(HERE, "liboracle_adaln.so")

FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
         "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra"]


def compile_oracle(src=SRC, out=LIB, extra=()):
    """Build `src` into the shared library `out` and return its path."""
    cmd = ["g++", *FLAGS, *extra, "-o", out, src]
    subprocess.run(cmd, check=True, cwd=HERE)
    return out


def build(force=False):
    """Build the oracle library if it is missing or older than its sources."""
    if not force and os.path.exists(LIB):
        lib_t = os.path.getmtime(LIB)
        if lib_t >= max(os.path.getmtime(SRC), os.path.getmtime(HDR)):
            return LIB
    return compile_oracle()


if __name__ == "__main__":
    print(build(force=True))
