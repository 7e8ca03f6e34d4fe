"""The C ABI from a C program: gcc compiles tests/c_abi/abi_from_c.c against include/gdn.h and links
libgdn.so; the program checks host-side validation (no GPU needed)."""
import os
import subprocess

import pytest

from gated_deltanet_linear_mtp_gb300 import build as gbuild

HERE = os.path.dirname(os.path.abspath(__file__))


def test_c_caller(tmp_path):
    if not os.path.exists(gbuild.LIB_PATH):
        gbuild.build()
    exe = tmp_path / "abi_from_c"
    libdir = os.path.dirname(gbuild.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", f"-I{gbuild.INCLUDE}", os.path.join(HERE, "c_abi", "abi_from_c.c"),
                    f"-L{libdir}", "-lgdn", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "abi_from_c: ok" in r.stdout
