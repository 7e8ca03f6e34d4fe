"""The C ABI from C programs: gcc compiles them against include/gdn.h and links libgdn.so.

* ``abi_from_c.c`` checks host-side validation and status strings (no GPU needed).
* ``verify_commit_from_c.c`` allocates device buffers itself, copies the tiny fp32 workload in from host arrays,
  calls gdn_mtp_verify + gdn_commit and checks the results against oracle values this test writes beside the
  inputs (GPU).
* ``in_proj_from_c.c`` does the same for gdn_in_proj_conv (decode rows) (GPU)."""
import os
import subprocess

import numpy as np
import pytest

import gdn_workloads as W
import oracle
from gated_deltanet_linear_mtp_gb300 import build as gbuild

HERE = os.path.dirname(os.path.abspath(__file__))
LIBDIR = os.path.dirname(gbuild.LIB_PATH)


def _lib():
    if not os.path.exists(gbuild.LIB_PATH):
        gbuild.build()


def _cuda_dirs():
    home = os.path.dirname(os.path.dirname(os.path.realpath(gbuild.nvcc())))
    return os.path.join(home, "include"), os.path.join(home, "lib64")


def _compile(src: str, exe, cuda: bool):
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", f"-I{gbuild.INCLUDE}"]
    if cuda:
        inc, lib = _cuda_dirs()
        cmd += [f"-I{inc}"]
    cmd += [os.path.join(HERE, "c_abi", src), f"-L{LIBDIR}", "-lgdn", f"-Wl,-rpath,{LIBDIR}"]
    if cuda:
        cmd += [f"-L{lib}", "-lcudart", f"-Wl,-rpath,{lib}", "-lm"]
    subprocess.run(cmd + ["-o", str(exe)], check=True)


def test_c_caller(tmp_path):
    _lib()
    exe = tmp_path / "abi_from_c"
    _compile("abi_from_c.c", exe, cuda=False)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "abi_from_c: ok" in r.stdout


def test_c_launcher_compiles(tmp_path):
    """The launching C program builds against the CUDA runtime headers (run on the GPU below)."""
    _lib()
    _compile("verify_commit_from_c.c", tmp_path / "verify_commit_from_c", cuda=True)


def _write_inputs(dirpath, w):
    x = w.arrays()
    o_ref, c_ref, flags = oracle.default().verify(oracle.dims_of(w), x, cache=True)
    assert flags == 0
    with open(os.path.join(dirpath, "dims.txt"), "w") as f:
        f.write(f"{w.B} {w.T} {w.HK} {w.HV} {w.DK} {w.DV} {w.num_slots}\n")
    for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "pool"):
        np.ascontiguousarray(x[k], dtype=np.float32).tofile(os.path.join(dirpath, f"{k}.bin"))
    for k in ("indices", "accept_len"):
        np.ascontiguousarray(x[k], dtype=np.int32).tofile(os.path.join(dirpath, f"{k}.bin"))
    np.ascontiguousarray(o_ref, dtype=np.float64).tofile(os.path.join(dirpath, "o_ref.bin"))
    np.ascontiguousarray(c_ref, dtype=np.float32).tofile(os.path.join(dirpath, "cache_ref.bin"))


@pytest.mark.gpu
@pytest.mark.parametrize("w", [W.tiny(), W.tiny().replace(name="small_B5_T3_d32_f32", B=5, T=3, HK=2, HV=4, DK=32,
                                                          DV=40, num_slots=9, seed=31, pad_fraction=0.2)],
                         ids=lambda w: w.name)
def test_c_program_runs_verify_and_commit(tmp_path, w):
    _lib()
    exe = tmp_path / "verify_commit_from_c"
    _compile("verify_commit_from_c.c", exe, cuda=True)
    data = tmp_path / "data"
    data.mkdir()
    _write_inputs(str(data), w)
    r = subprocess.run([str(exe), str(data)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "verify_commit_from_c: ok" in r.stdout


def test_c_in_proj_launcher_compiles(tmp_path):
    """The in_proj C program builds against the CUDA runtime headers (run on the GPU below)."""
    _lib()
    _compile("in_proj_from_c.c", tmp_path / "in_proj_from_c", cuda=True)


def _write_in_proj_inputs(dirpath, w):
    x = w.arrays()
    d = dict(T=w.T, H=w.H, HK=w.HK, HV=w.HV, DK=w.DK, DV=w.DV, K=w.K, num_slots=w.num_slots, x_dtype="bf16",
             conv_dtype="bf16", silu=1)
    state_ref = x["conv_state"].copy()
    out_ref, _, flags = oracle.default().in_proj_conv(d, x["x"], x["W"], x["conv_w"], x["conv_b"], state_ref,
                                                      x["indices"], write_pool=True, records=False)
    assert flags == 0
    with open(os.path.join(dirpath, "dims.txt"), "w") as f:
        f.write(f"{w.B} {w.T} {w.H} {w.HK} {w.HV} {w.DK} {w.DV} {w.K} {w.num_slots}\n")
    for k, name in (("x", "x"), ("W", "W"), ("conv_state", "state")):
        np.ascontiguousarray(x[k], dtype=np.uint16).tofile(os.path.join(dirpath, f"{name}.bin"))
    for k in ("conv_w", "conv_b"):
        np.ascontiguousarray(x[k], dtype=np.float32).tofile(os.path.join(dirpath, f"{k}.bin"))
    np.ascontiguousarray(x["indices"], dtype=np.int32).tofile(os.path.join(dirpath, "indices.bin"))
    np.ascontiguousarray(out_ref, dtype=np.float64).tofile(os.path.join(dirpath, "out_ref.bin"))
    np.ascontiguousarray(state_ref, dtype=np.uint16).tofile(os.path.join(dirpath, "state_ref.bin"))


@pytest.mark.gpu
def test_c_program_runs_in_proj(tmp_path):
    """A plain C program runs the in_proj projection with its conv1d epilogue (decode rows) on buffers it copied in
    from the host, one lane padded, and checks the outputs and the written-back state against the oracle."""
    _lib()
    exe = tmp_path / "in_proj_from_c"
    _compile("in_proj_from_c.c", exe, cuda=True)
    data = tmp_path / "data"
    data.mkdir()
    w = W.InProjWorkload("c_in_proj", B=3, T=2, H=128, HK=1, HV=2, DK=16, DV=16, K=4, num_slots=6,
                         conv_dtype="bf16", out_dtype="f32", seed=33, pad_fraction=0.34)
    _write_in_proj_inputs(str(data), w)
    r = subprocess.run([str(exe), str(data)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "in_proj_from_c: ok" in r.stdout
