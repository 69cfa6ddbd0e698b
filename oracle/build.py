"""Compile the CPU oracle (oracle.c) into oracle/_build/liboracle.so.

Test infrastructure only: only tests/, __graft_entry__ and bench.py's CPU
baseline leg load the result.  gcc with OpenMP when the compiler supports it,
serial otherwise (results are identical either way).
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def _has_openmp(cc: str) -> bool:
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        with open(src, "w") as f:
            f.write("#include <omp.h>\nint main(void){return omp_get_max_threads() > 0 ? 0 : 1;}\n")
        r = subprocess.run([cc, "-fopenmp", src, "-o", os.path.join(d, "t")],
                           capture_output=True)
        return r.returncode == 0


def build(force: bool = False) -> str:
    src = os.path.join(HERE, "oracle.c")
    hdr = os.path.join(HERE, "oracle.h")
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(src), os.path.getmtime(hdr))):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    flags = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-Wall"]
    if _has_openmp(cc):
        flags.append("-fopenmp")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *flags, src, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + " ".join(cmd) + "\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
