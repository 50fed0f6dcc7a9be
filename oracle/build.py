"""Compile the fp64 CPU oracle (``ea_oracle.c``) into ``oracle/_build/libea_oracle.so``.

Test infrastructure: the oracle is only ever loaded by the tests, the package's
smoke check and the benchmark's CPU-baseline leg.  Plain gcc, OpenMP when the
compiler has it; no architecture-specific flags, so the same source builds on
x86_64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ea_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "libea_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(SRC), os.path.getmtime(os.path.abspath(__file__)))
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= newest:
        return OUT
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", "-ffp-contract=off", SRC,
            "-lm"]
    tmp = OUT + ".tmp.%d" % os.getpid()
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:] + ["-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, OUT)
            if verbose:
                print(" ".join(cmd))
            return OUT
    raise RuntimeError("oracle build failed:\n" + r.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
