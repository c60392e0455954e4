"""Compile the fp64 CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, OpenMP when the compiler has it, -ffp-contract=off so that the
same source gives the same bits on x86-64 and aarch64 hosts.  Nothing here
is used by the CUDA library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "wanvae_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-std=c11", "-O3", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-fvisibility=hidden", SRC, "-o", LIB + ".tmp", "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(LIB + ".tmp", LIB)
            if verbose:
                print(" ".join(cmd))
            return LIB
    raise RuntimeError("oracle build failed:\n" + r.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
