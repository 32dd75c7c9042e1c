"""Build the C part of the oracle (attn_ref.c, pack_ref.c) into
oracle/_build/liboracle.so with the host gcc and OpenMP. TEST INFRASTRUCTURE
ONLY; compiled by __graft_entry__.build() so the checker exists wherever the
tests run. Plain C, no architecture-specific flags, so it builds the same on
x86_64 and aarch64 hosts."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")
SOURCES = [os.path.join(HERE, "attn_ref.c"), os.path.join(HERE, "pack_ref.c")]


def build(force=False):
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        lib_m = os.path.getmtime(LIB)
        if all(os.path.getmtime(s) <= lib_m for s in SOURCES):
            return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp] + SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
