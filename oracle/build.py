"""Compile the CPU oracle (oracle.c) into oracle/liboracle.so.

Test infrastructure: the oracle is only loaded by tests/, by
``__graft_entry__.smoke()`` and by the cpu_baseline / reference legs of
bench.py.  Building it is not using it: ``__graft_entry__.build()`` compiles it
next to the CUDA library so that the checker exists on every machine.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def is_stale() -> bool:
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    """Build liboracle.so with gcc (plain C11, no fp contraction)."""
    if force or is_stale():
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-Wall", "-Wextra", "-Wno-unused-parameter",
               "-shared", "-fPIC", "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
