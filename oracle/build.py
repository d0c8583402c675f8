"""Build the CPU oracle (test infrastructure) as a shared library with gcc.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg use
the result.  Flags keep IEEE semantics: no fast-math, no FP contraction, so the
FP32 mirror's fmaf/addition sequence is exactly the one written in the source.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")
SOURCES = [os.path.join(HERE, s) for s in ("oracle.c", "mirror.c")]


def build(force: bool = False) -> str:
    """Compile oracle.c and mirror.c into _build/liboracle.so; return its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(s) for s in SOURCES)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           "-o", tmp, *SOURCES, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
