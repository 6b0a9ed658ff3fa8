"""Compile the oracle (plain C) into ``oracle/liboracle.so`` with gcc.

Test infrastructure: building the checker is not using it.  The flags keep
every float operation a single IEEE binary32 operation: no fast-math and no
contraction of a multiply and an add into one fused operation.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


SELFTEST_SRC = os.path.join(HERE, "selftest.c")
SELFTEST = os.path.join(HERE, "selftest")


def _fresh(out, *srcs):
    return os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(s) for s in srcs)


def build(force: bool = False) -> str:
    """liboracle.so, and the C self-test program linked against it."""
    if force or not _fresh(LIB, SRC):
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
               "-fexcess-precision=standard", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    if force or not _fresh(SELFTEST, SELFTEST_SRC, LIB):
        tmp = SELFTEST + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O1", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra",
               "-o", tmp, SELFTEST_SRC, "-L", HERE, "-loracle", "-Wl,-rpath," + HERE, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, SELFTEST)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
