"""Build the CPU oracle shared library (TEST INFRASTRUCTURE ONLY).

    python -m oracle.build        # -> oracle/_build/libtq_oracle.so

Plain gcc, -O2 -ffp-contract=off (every float op rounds once, in source
order), OpenMP when the compiler has it.  No architecture flags, so the same
source gives the same results on x86-64 and aarch64.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libtq_oracle.so")
SOURCES = [os.path.join(HERE, "tq_oracle.c")]


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = SOURCES + [os.path.join(HERE, "tq_oracle.h"), os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            *SOURCES, "-o", LIB_PATH + ".tmp", "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(LIB_PATH + ".tmp", LIB_PATH)
            if verbose:
                print(" ".join(cmd))
            return LIB_PATH
        last = r
    raise RuntimeError(f"oracle build failed:\n{last.stderr}")


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
