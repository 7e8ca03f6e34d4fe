"""Register spills of the timed kernels, from ptxas's own report (``-Xptxas -v``, no GPU needed): the kernels
the benchmarks time keep their state in registers, so a change that makes one of them spill (a new live
value, a changed launch bound) fails here before it costs bandwidth on the GPU.  Ceilings are the spills
measured when the kernels were timed: none, except 4 bytes (outside the token loop's hot path) in the
16 KiB bulk-copy kernel."""
import os
import re
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

from gated_deltanet_linear_mtp_gb300 import build as gbuild

# (source, substring of the mangled kernel name, spill-store ceiling in bytes)
TIMED = [
    ("gdn_recurrent_bf16.cu", "gdn_recurrent_staged_kernelILi128E13__nv_bfloat16S1_Li16ELb0E", 4),  # verify T=4
    ("gdn_recurrent_bf16.cu", "gdn_recurrent_staged_kernelILi128E13__nv_bfloat16S1_Li32ELb0E", 0),  # bf16 T <= 2
    ("gdn_recurrent_bf16.cu", "gdn_recurrent_kernelILi128E13__nv_bfloat16S1_Lb0E", 0),              # verify T=8
    ("gdn_recurrent_bf16.cu", "gdn_recurrent_staged_kernelILi128E13__nv_bfloat16S1_Li32ELb1E", 0),  # decode + norm
    ("gdn_recurrent_bf16.cu", "gdn_recurrent_kernelILi128E13__nv_bfloat16S1_Lb1E", 0),              # small B + norm
    ("gdn_recurrent_bf16.cu", "gdn_verify_chunked_kernelILi128E13__nv_bfloat16Li0E", 0),          # verify, no cache
    ("gdn_recurrent_bf16.cu", "gdn_verify_chunked_kernelILi128E13__nv_bfloat16Li1E", 0),          # replay commit
    ("gdn_recurrent_bf16.cu", "gdn_verify_chunked_kernelILi128E13__nv_bfloat16Li2E", 0),          # one-pass step
    ("gdn_recurrent_f32.cu", "gdn_recurrent_staged_kernelILi128E13__nv_bfloat16fLi16ELb0E", 0),   # decode fp32
    ("gdn_prefill.cu", "gdn_prefill_kernelILi256E13__nv_bfloat16S1_E", 0),                        # prefill token loop (DK 16, 32, 256)
    ("gdn_prefill_chunked.cu", "gdn_prefill_chunked_kernelILi128E13__nv_bfloat16S2_Lb1E", 0),     # prefill (TMA)
    ("gdn_prefill_chunked.cu", "gdn_prefill_chunked_kernelILi128EffLb0E", 0),                     # prefill fp32
    ("gdn_gated_norm.cu", "gdn_gated_rmsnorm_reg_kernel", 0),                                    # gated norm
    ("gdn_in_proj_conv.cu", "gdn_in_proj_conv_kernelILi4E", 0),                                  # in_proj + conv1d
    ("gdn_in_proj_conv.cu", "gdn_conv_commit_kernel", 0),                                        # conv state commit
]


def ptxas_spills(src: str):
    """{mangled kernel name: spill-store bytes} of one translation unit."""
    cmd = [gbuild.nvcc(), *gbuild.NVCC_FLAGS, "-Xptxas", "-v", "-c", os.path.join(gbuild.CSRC, src), "-o",
           os.devnull]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out, cur = {}, None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores", line)
        if m and cur is not None:
            out[cur] = int(m.group(1))
            cur = None
    return out


@pytest.fixture(scope="module")
def spills():
    try:
        gbuild.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    srcs = sorted({s for s, _, _ in TIMED})
    with ThreadPoolExecutor(len(srcs)) as ex:
        return dict(zip(srcs, ex.map(ptxas_spills, srcs)))


@pytest.mark.parametrize("src,kernel,ceiling", TIMED, ids=[k for _, k, _ in TIMED])
def test_timed_kernels_do_not_spill(spills, src, kernel, ceiling):
    found = {name: b for name, b in spills[src].items() if kernel in name}
    assert found, f"no kernel matching {kernel} in {src}"
    worst = max(found.values())
    assert worst <= ceiling, f"{kernel}: {worst} bytes of spill stores (ceiling {ceiling})"
