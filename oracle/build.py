"""Compile the C oracle into ``oracle/_build/liboracle.so`` (test infrastructure only).

Plain gcc, fp64, OpenMP, and ``-ffp-contract=off`` so that no fused multiply-add
changes the rounding between the x86 and Arm hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")
SOURCES = ["attn_oracle.c"]
DEPS = SOURCES + ["tiled_body.h"]


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t for s in DEPS)


def build(force: bool = False, defines: tuple[str, ...] = (), out: str | None = None) -> str:
    """Build the oracle library; returns its path.  ``defines`` is for tests only."""
    out = out or LIB_PATH
    if not force and out == LIB_PATH and not _stale():
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           *[f"-D{d}" for d in defines],
           *[os.path.join(HERE, s) for s in SOURCES], "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
