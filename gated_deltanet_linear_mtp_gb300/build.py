"""Builds ``libgdn.so`` in-tree for sm_103a with nvcc (one -gencode, translation units in parallel).

    python -m gated_deltanet_linear_mtp_gb300.build

The CUDA runtime is linked statically, so the library needs only the driver at run time and loads (for
its host-side argument checks) on a machine without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libgdn.so")

SOURCES = ["gdn_api.cu", "gdn_recurrent_f32.cu", "gdn_recurrent_bf16.cu", "gdn_commit.cu", "gdn_prefill.cu",
           "gdn_prefill_chunked.cu", "gdn_gated_norm.cu", "gdn_in_proj_conv.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# hidden visibility: only the GDN_API functions of gdn.h are exported, so that internal symbols (template
# statics among them) never bind across two libraries loaded in one process
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-cudart", "static", f"-I{INCLUDE}", f"-I{CSRC}"] + ARCH
LINK_FLAGS = ["-shared", "-cudart", "static", "-Xlinker", "--exclude-libs=ALL"]  # nor the static runtime's


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn.so")


def _compile(src: str, extra: List[str], obj_dir: str) -> str:
    obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(extra: List[str] = (), out_dir: Optional[str] = None) -> str:
    """Compile and link the library: in-tree by default; into `out_dir` (objects and libgdn.so) for a build
    with other flags, e.g. the wait-timeout test build of tests/test_gpu_timeout.py."""
    obj_dir = OBJ_DIR if out_dir is None else os.path.join(out_dir, "obj")
    lib_path = LIB_PATH if out_dir is None else os.path.join(out_dir, "libgdn.so")
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra), obj_dir), SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [nvcc(), *LINK_FLAGS, *ARCH, *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(sys.argv[1:]))
