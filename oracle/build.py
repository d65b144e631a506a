"""Compile the float64 CPU oracle (test infrastructure) with the host C compiler.

The shared object lands next to the source as ``libspec_oracle.so``; a stamp
file holding the source hash makes repeated builds free.
"""
from __future__ import annotations

import hashlib
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spec_oracle.c")
LIB = os.path.join(HERE, "libspec_oracle.so")
STAMP = LIB + ".stamp"


def _digest() -> str:
    with open(SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def build(force: bool = False) -> str:
    """Build the oracle library if missing or stale; return its path."""
    digest = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == digest:
                return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -O2 without -ffast-math: the oracle keeps IEEE float64 semantics.
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
