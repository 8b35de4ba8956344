"""Compile the C oracle (test infrastructure only) with the host gcc.

The shared object goes to ``oracle/_build/``.  A mutation build (a copy with
one planted mistake, used only by the test that shows the pins catch it) gets
its own file name.
"""
from __future__ import annotations

import os
import subprocess
import sys
from pathlib import Path

HERE = Path(__file__).resolve().parent
SRC = HERE / "ssd_oracle.c"
OUT_DIR = HERE / "_build"


def lib_path(mutation: int = 0) -> Path:
    suffix = "" if mutation == 0 else f"_mut{mutation}"
    return OUT_DIR / f"libssd_oracle{suffix}.so"


def build(mutation: int = 0, force: bool = False) -> Path:
    out = lib_path(mutation)
    if out.exists() and not force and out.stat().st_mtime >= SRC.stat().st_mtime:
        return out
    OUT_DIR.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".tmp{os.getpid()}.so")
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC",
            f"-DSSD_ORACLE_MUTATION={mutation}", str(SRC), "-o", str(tmp), "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # no OpenMP runtime: the pragma is ignored and the oracle runs serially
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(int(sys.argv[1]) if len(sys.argv) > 1 else 0, force=True))
