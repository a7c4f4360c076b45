"""Build the C part of the oracle (the fp32 contract emulator) in place.

TEST INFRASTRUCTURE ONLY.  Produces oracle/libcontract_emulator.so with gcc.
``-ffp-contract=off`` keeps the compiler from fusing a*b+c on its own (gcc
fuses by default on aarch64), so the only fused multiply-adds are the
explicit ``fmaf`` calls the contract names.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "contract_emulator.c")
LIB = os.path.join(HERE, "libcontract_emulator.so")

CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-fopenmp", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc"] + CFLAGS + ["-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
