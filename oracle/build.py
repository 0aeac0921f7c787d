"""Compile the C oracle into oracle/_build/libpa_oracle.so with gcc.

Test infrastructure only: the library it makes is loaded by tests/, by the
smoke check and by bench.py's CPU-baseline / reference legs, never by the
product path.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpa_oracle.so")


def command():
    # Plain -O2: no -ffast-math (it would reorder the fp64 sums and break the
    # IEEE special cases the widening relies on), no machine-specific flags so
    # the same source gives the same results on x86_64 and aarch64.
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
            "-o", LIB, SRC, "-lm"]


def start():
    """Start the compile and return the Popen (so callers can overlap it)."""
    os.makedirs(OUT_DIR, exist_ok=True)
    return subprocess.Popen(command(), stdout=subprocess.PIPE, stderr=subprocess.STDOUT)


def build():
    p = start()
    out, _ = p.communicate()
    if p.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + out.decode(errors="replace"))
    return LIB


def is_stale():
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


if __name__ == "__main__":
    print(build())
    sys.exit(0)
