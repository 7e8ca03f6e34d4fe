"""The bounded waits of the copy-fed kernels, made to run out without a fault.

A test build of the library (flags GDN_TEST_MISSING_COPY and a short GDN_WAIT_POLLS) leaves one bulk / TMA
copy unissued and never arrives on its mbarrier, so the wait for it can only run out (the staged and chunked
verify, the replay commit, the chunked prefill, the in_proj + conv1d kernel).  That is the same path
a copy that never lands would take: the kernel sets GDN_ERRBIT_TIMEOUT, gives up the work it waited for,
drains the copies it did issue and ends.  Nothing is left in flight, so the GPU context stays usable: the
product library then runs a normal call in the same process and matches the oracle."""
import os

import numpy as np
import pytest
import torch

import gated_deltanet_linear_mtp_gb300 as gdn
import gdn_workloads as W
from gated_deltanet_linear_mtp_gb300 import build as gbuild
from gpu_util import Dev, dev, host, run_verify
from test_gpu_parity import compare_verify

pytestmark = pytest.mark.gpu

TEST_BUILD = os.path.join(gbuild.PKG, "_build", "wait_timeout_test")


@pytest.fixture(scope="module")
def timeout_lib():
    return gbuild.build(["-DGDN_TEST_MISSING_COPY", "-DGDN_WAIT_POLLS=65536u"], out_dir=TEST_BUILD)


def workload(name, T, cache, **kw):
    # lane 0 active (the missing copy belongs to lane 0, head 0, rows 0..); enough CTAs for the staged kernel
    base = dict(B=8, HK=16, HV=48, DK=128, DV=128, num_slots=10, qkv_dtype="bf16", state_dtype="bf16",
                out_dtype="bf16", mode="verify", cache=cache, commit=True, seed=21, pool_std=0.1)
    base.update(kw)
    return W.Workload(name, T=T, **base)


def run_with(lib_path, monkeypatch, fn):
    monkeypatch.setattr(gdn, "_lib_handle", None)
    monkeypatch.setattr(gdn, "LIB_PATH", lib_path)
    try:
        return fn()
    finally:
        monkeypatch.setattr(gdn, "_lib_handle", None)
        monkeypatch.setattr(gdn, "LIB_PATH", gbuild.LIB_PATH)


@pytest.mark.parametrize("case", ["chunked_verify", "chunked_replay", "staged_verify"])
def test_wait_that_runs_out_sets_the_timeout_bit(timeout_lib, monkeypatch, case):
    if case == "staged_verify":  # bf16, T = 2, with the cache: the staged (bulk-copy) kernel
        w = workload("timeout_staged", T=2, cache=True)
    else:  # bf16, T = 4, no cache: the chunked (TMA) kernel
        w = workload("timeout_chunked", T=4, cache=False)
    x = w.arrays()
    x["indices"][0] = 0 if x["indices"][0] < 0 else x["indices"][0]
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        if case == "chunked_replay":  # into a copy: the pool itself must stay as the oracle has it
            pool = t["pool"].clone()
            gdn.gdn_commit_replay(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], pool,
                                  t["indices"], t["accept_len"], err, scale=w.scale, l2_eps=w.l2_eps)
        else:
            run_verify(w, t, cache=w.cache, err=err)
        torch.cuda.synchronize()

    run_with(timeout_lib, monkeypatch, call)
    assert int(err.item()) & gdn.ERRBIT_TIMEOUT, "the wait did not report running out"

    # the context is usable: the product library verifies the same batch correctly afterwards
    err.zero_()
    o, cache = run_verify(w, t, cache=w.cache, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    lanes = np.flatnonzero(x["indices"] >= 0)[:4]
    compare_verify(w, x, host(o), host(cache) if cache is not None else None, lanes=lanes)


def test_chunked_prefill_wait_that_runs_out(timeout_lib, monkeypatch):
    """The chunked prefill (bf16 tokens by TMA): the first chunk of its first item is never loaded, so the token
    group's wait for it runs out, and then the row group's wait for that chunk; the bit is set, the CTA drains
    the loads it did issue and ends, and the product library then prefills the batch correctly."""
    from test_gpu_prefill import compare_prefill, run_prefill, small
    pw = small("timeout_prefill", [70, 40], DK=128, DV=128, HK=1, HV=2, seed=23, fresh=0.0)
    x = pw.arrays()
    t = Dev(x)
    before = host(t["pool"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():  # into a copy of the pool: the product run below starts from the untouched one
        tt = {k: t[k] for k in x}
        tt["pool"] = t["pool"].clone()
        run_prefill(pw, tt, err)
        torch.cuda.synchronize()

    run_with(timeout_lib, monkeypatch, call)
    assert int(err.item()) & gdn.ERRBIT_TIMEOUT, "the wait did not report running out"
    err.zero_()
    o = run_prefill(pw, t, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    compare_prefill(pw, x, host(o), host(t["pool"]), before)


def test_in_proj_wait_that_runs_out(timeout_lib, monkeypatch):
    """The in_proj + conv1d kernel (W by TMA, the hidden dimension split over a cluster): the first stage of the
    first CTA is never loaded, so its MMA thread's wait runs out, then the producer's wait for the stage to come
    free; the bit is set, the CTA drains the loads it did issue, every rank of the cluster still meets at its
    barriers, and the product library then computes the batch correctly."""
    from test_gpu_in_proj_conv import check_call, outputs, small
    w = small("timeout_in_proj", B=4, T=4, H=512, seed=25)
    x = w.arrays()
    t = {k: dev(v) for k, v in x.items()}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        rec = torch.zeros((w.B, w.T, w.Cc), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_in_proj_conv(t["x"], t["W"], t["conv_w"], t["conv_b"], t["conv_state"], t["indices"], outputs(w),
                             False, rec, err)
        torch.cuda.synchronize()

    run_with(timeout_lib, monkeypatch, call)
    assert int(err.item()) & gdn.ERRBIT_TIMEOUT, "the wait did not report running out"
    check_call(w, x, False)
