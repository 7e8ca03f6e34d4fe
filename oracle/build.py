"""Compiles the C oracle (``gdn_oracle.c``) with gcc into a shared library.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  ``-ffp-contract=off`` keeps every multiply and add
separately rounded, so x86 and Arm builds give the same bits.  No ``-ffast-math``: IEEE semantics.
"""
from __future__ import annotations

import os
import subprocess
import sys
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "gdn_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
CFLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra"]


def library_path() -> str:
    return os.path.join(BUILD_DIR, "libgdn_oracle.so")


def build(source: Optional[str] = None, out: Optional[str] = None, extra: Sequence[str] = ()) -> str:
    """Compile ``source`` (default: the committed oracle) to ``out``; returns the library path."""
    source = source or SOURCE
    out = out or library_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, *extra, source, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(*sys.argv[1:2]))
