"""Compile the fp64 CPU oracle (``gdn_oracle.c``) into ``oracle/_build/libgdn_oracle.so``.

Test infrastructure: the oracle is built here so that the tests, the smoke
check and the bench's CPU-baseline leg can load it.  Plain gcc, no CUDA.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libgdn_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    # -ffp-contract=off: every product and sum is rounded as written (no FMA
    # fusion), so the x86 and Arm builds give the same doubles.
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
