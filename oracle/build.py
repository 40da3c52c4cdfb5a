"""Build the fp64 CPU oracle (test infrastructure) into oracle/_build/liboracle.so.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use the
result.  Portable flags only: the same source must give the same numbers on
x86-64 and aarch64, so floating-point contraction is disabled (an FMA would
change the rounding of the fp64 arithmetic) and no -march is given.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "liboracle.so")


def _cmd(openmp):
    flags = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter"]
    if openmp:
        flags.append("-fopenmp")
    return flags + [SRC, "-o", OUT, "-lm"]


def build(force=False, verbose=False):
    """Compile the oracle if the shared object is missing or older than the source."""
    if (not force and os.path.exists(OUT)
            and os.path.getmtime(OUT) >= os.path.getmtime(SRC)):
        return OUT
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = OUT + ".tmp%d" % os.getpid()
    for openmp in (True, False):
        cmd = _cmd(openmp)
        cmd[cmd.index(OUT)] = tmp
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, OUT)
            if verbose and r.stderr:
                print(r.stderr, file=sys.stderr)
            return OUT
        last = r
    raise RuntimeError("oracle build failed:\n" + last.stderr)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
