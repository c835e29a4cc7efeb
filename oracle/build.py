"""Build the CPU oracle (test infrastructure) as oracle/_build/libdsoracle.so.

Plain C++17, no vectorisation flags and no fused multiply-add contraction, so
that the same source gives the same results on x86-64 and aarch64.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libdsoracle.so")
SOURCES = [os.path.join(HERE, "dsoracle.cpp")]


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its sources; return the .so path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    deps = SOURCES + [os.path.join(HERE, "dsoracle.h")]
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(p) for p in deps):
            return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp] + SOURCES
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
