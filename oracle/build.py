"""Compile the CPU oracle into oracle/libsrwm_oracle.so with the host C compiler.

TEST INFRASTRUCTURE: the oracle is a checker, never part of the product path.
Building it here makes it available to the tests, the smoke check and the
benchmark's CPU-baseline leg on whatever machine they run.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = [os.path.join(HERE, "srwm_oracle.c"), os.path.join(HERE, "srwm_oracle_core.h")]
LIB = os.path.join(HERE, "libsrwm_oracle.so")


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in SOURCES)


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its sources."""
    if not force and not is_stale():
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    # -O2 without -ffast-math: no reassociation, so each sum runs in source order.
    cmd = [cc, "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, SOURCES[0], "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
