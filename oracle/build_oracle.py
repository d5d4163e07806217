"""Compile the C oracle (forward and backward) into ``oracle/lib/libkda_oracle.so`` (test
infrastructure only).

Plain gcc, no architecture-specific flags, so that the same source builds on x86_64 and
aarch64 hosts. ``-ffp-contract=off`` keeps every fp64 multiply and add separately
rounded, as the source states them.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "kda_oracle.c"), os.path.join(HERE, "kda_oracle_bwd.c")]
LIB_DIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIB_DIR, "libkda_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if not force and os.path.exists(LIB) and all(os.path.getmtime(LIB) >= os.path.getmtime(s) for s in SRCS):
        return LIB
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-Wall", "-Wextra", "-o", tmp, *SRCS, "-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
