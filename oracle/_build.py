"""Builds the oracle (plain C, f64, single-threaded) in-tree as liboracle.so.

Building the checker is not using it: the library is loaded only by the test
suite, the package smoke check and the benchmark's CPU-baseline leg.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(HERE, "liboracle.so")


def build(force=False):
    srcs = [os.path.join(HERE, "moe_oracle.c"), os.path.join(HERE, "moe_oracle.h")]
    stale = (not os.path.exists(SO)) or any(os.path.getmtime(s) > os.path.getmtime(SO) for s in srcs)
    if force or stale:
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math", "-fvisibility=hidden",
                               "-o", SO, srcs[0], "-lm"])
    return SO


if __name__ == "__main__":
    build(force=True)
