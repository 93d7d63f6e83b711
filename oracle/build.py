"""Build the CPU oracle (``liborc.so``) with the system C compiler.

Test infrastructure only: the oracle checks the CUDA library and is never
linked into it.  OpenMP is used when the compiler supports it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pskv_oracle.c")
LIB = os.path.join(HERE, "liborc.so")


def _compile(out: str, extra: list[str]) -> subprocess.CompletedProcess:
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-Wno-unused-parameter", *extra, SRC, "-o", out, "-lm"]
    return subprocess.run(cmd, capture_output=True, text=True)


def build(force: bool = False, out: str = LIB) -> str:
    """Compile the oracle if it is missing or older than its source; return the path."""
    srcs = [SRC, os.path.join(HERE, "pskv_oracle.h")]
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(s) for s in srcs)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    res = _compile(tmp, ["-fopenmp"])
    if res.returncode != 0:  # no OpenMP on this compiler: build serial
        res = _compile(tmp, [])
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
