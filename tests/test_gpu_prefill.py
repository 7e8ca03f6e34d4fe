"""Parity of the prefill call (``gdn_prefill``) and the gated RMSNorm (``gdn_gated_rmsnorm``) with the CPU
oracle, through the C ABI, on seeded inputs.

Prefill: variable-length sequences that span several token chunks with ragged tails, empty sequences,
padded (-1) lanes, sequences with and without an initial state (a fresh slot holds NaN and must not be
read), every DK, both state and input types, a ragged DV; at the ISL-8K size on sampled (sequence, head)
pairs the oracle runs one at a time.  Gated norm: every lane-group width of the vector path, the
column-at-a-time path (ragged DV, misaligned rows), in place, and after a verify call.  Tolerances: see
``gpu_util``.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gated_deltanet_linear_mtp_gb300 as gdn
import gdn_workloads as W
import oracle
from gpu_util import (Dev, assert_f32_close, canary, check_o, check_state, dev, host,
                      is_canary, run_verify, storage_to_f64)

pytestmark = pytest.mark.gpu


def prefill_dims(pw) -> dict:
    return dict(T=0, HK=pw.HK, HV=pw.HV, DK=pw.DK, DV=pw.DV, num_slots=pw.num_slots, qkv_dtype=pw.qkv_dtype,
                state_dtype=pw.state_dtype, scale=pw.scale, l2_eps=pw.l2_eps)


def run_prefill(pw, t: Dev, err=None, o=None, has_init=True):
    N = t["q"].shape[0]
    if o is None:
        o = canary((N, pw.HV, pw.DV), pw.out_dtype)
    gdn.gdn_prefill(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"],
                    t["cu_seqlens"], o, t["has_initial_state"] if has_init else None, err, scale=pw.scale,
                    l2_eps=pw.l2_eps)
    return o


def compare_prefill(pw, x, o_gpu, pool_gpu, pool_before, has_init=True):
    """o at every token and the pool (every slot) against the oracle; skipped sequences keep their canaries."""
    orc = oracle.default()
    pool_ref = x["pool"].copy()
    o_ref, fl = orc.prefill(prefill_dims(pw), x, x["cu_seqlens"], pool_ref,
                            x["has_initial_state"] if has_init else None)
    cu, idx = x["cu_seqlens"], x["indices"]
    written = np.zeros(o_gpu.shape[0], bool)
    for b in range(pw.B):
        if 0 <= idx[b] < pw.num_slots and 0 <= cu[b] <= cu[b + 1] <= o_gpu.shape[0]:
            written[cu[b]:cu[b + 1]] = True
    if written.any():
        check_o(pw, o_gpu[written], o_ref[written], "prefill o")
    assert is_canary(o_gpu[~written]).all(), "o written outside the active sequences"
    touched = np.zeros(pw.num_slots, bool)
    for b in range(pw.B):
        s = idx[b]
        if 0 <= s < pw.num_slots and 0 <= cu[b] < cu[b + 1] <= o_gpu.shape[0]:
            touched[s] = True
    if touched.any():
        check_state(pw, pool_gpu[touched], pool_ref[touched], "prefill final state")
    assert np.array_equal(pool_gpu[~touched], pool_before[~touched]), "an untouched slot changed"
    return fl


def small(name, lengths, DK=128, DV=96, HK=2, HV=4, qkv="bf16", state="bf16", out=None, seed=11, pad=0.0,
          fresh=0.5):
    return W.PrefillWorkload(name, B=len(lengths), HK=HK, HV=HV, DK=DK, DV=DV, num_slots=len(lengths) + 3,
                             qkv_dtype=qkv, state_dtype=state, out_dtype=out or qkv, seed=seed,
                             lengths=tuple(lengths), fresh_fraction=fresh, pad_fraction=pad, pool_std=0.1)


# ---------------------------------------------------------------------------------------------------------
def test_prefill_varlen_chunks_and_tails():
    # lengths around the 8-token chunk of DK = 128: 1, 7, 8, 9, 16, 17, 33, 64, and an empty sequence
    pw = small("prefill_varlen", [1, 7, 0, 33, 16, 17, 64, 8, 9], pad=0.12)
    x = pw.arrays()
    t = Dev(x)
    before = host(t["pool"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = run_prefill(pw, t, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert (x["indices"] == -1).sum() == 1 and (x["has_initial_state"] == 0).any()
    compare_prefill(pw, x, host(o), host(t["pool"]), before)


@pytest.mark.parametrize("DK", [16, 32, 64, 256])
@pytest.mark.parametrize("qkv,state", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f32", "bf16")])
def test_prefill_every_dk_and_dtype(DK, qkv, state):
    lengths = [3, 0, 21, 40, 1, 17]
    pw = small(f"prefill_dk{DK}_{qkv}_{state}", lengths, DK=DK, DV=40 if DK != 256 else 24, HK=1, HV=2, qkv=qkv,
               state=state, seed=100 + DK)
    x = pw.arrays()
    t = Dev(x)
    before = host(t["pool"])
    o = run_prefill(pw, t)
    torch.cuda.synchronize()
    compare_prefill(pw, x, host(o), host(t["pool"]), before)


def test_prefill_without_mask_reads_every_slot():
    pw = small("prefill_nomask", [5, 12, 30], fresh=0.0, seed=13)
    x = pw.arrays()
    t = Dev(x)
    before = host(t["pool"])
    o = run_prefill(pw, t, has_init=False)
    torch.cuda.synchronize()
    compare_prefill(pw, x, host(o), host(t["pool"]), before, has_init=False)


@pytest.mark.parametrize("state", ["bf16", "f32"])
def test_prefill_fresh_slot_is_never_read(state):
    """Fresh sequences start from zero: NaN in their slots changes nothing (the result equals the oracle's
    with those slots zeroed, and the oracle never reads them either)."""
    pw = small("prefill_fresh_nan", [9, 25, 4, 13], state=state, fresh=0.5, seed=14)
    x = pw.arrays()
    fresh = np.flatnonzero(x["has_initial_state"] == 0)
    assert fresh.size == 2
    nan_pool = x["pool"].copy()
    if state == "bf16":
        nan_pool[x["indices"][fresh]] = 0x7FC1
    else:
        nan_pool[x["indices"][fresh]] = np.nan
    xn = dict(x, pool=nan_pool)
    t = Dev(xn)
    before = host(t["pool"])
    o = run_prefill(pw, t)
    torch.cuda.synchronize()
    o_h, pool_h = host(o), host(t["pool"])
    assert np.all(np.isfinite(storage_to_f64(o_h)))
    compare_prefill(pw, xn, o_h, pool_h, before)


def test_prefill_bad_bounds_and_index_set_error_bits():
    pw = small("prefill_bad", [6, 10, 4], seed=15, fresh=0.0)
    x = pw.arrays()
    N = int(x["cu_seqlens"][-1])
    i1, i2 = int(x["indices"][1]), int(x["indices"][2])
    # decreasing bounds skip sequence 1 (sequence 0 is padded, so that sequence 2 overlaps no written one);
    # a negative start skips sequence 0; an end beyond N sequence 2; then an index beyond the pool
    for cu, idx, want in (([0, 6, 5, 20], [-1, i1, i2], gdn.ERRBIT_SEQLEN),
                          ([-2, 6, 16, 20], None, gdn.ERRBIT_SEQLEN),
                          ([0, 6, 16, N + 1], None, gdn.ERRBIT_SEQLEN),
                          (None, [0, pw.num_slots, -1], gdn.ERRBIT_INDEX)):
        xb = dict(x)
        if cu is not None:
            xb["cu_seqlens"] = np.array(cu, np.int32)
        if idx is not None:
            xb["indices"] = np.array(idx, np.int32)
        t = Dev(xb)
        before = host(t["pool"])
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        o = run_prefill(pw, t, err)
        torch.cuda.synchronize()
        assert int(err.item()) == want, (cu, idx, int(err.item()))
        fl = compare_prefill(pw, xb, host(o), host(t["pool"]), before)
        assert fl == want


def test_prefill_host_checks():
    pw = small("prefill_host", [4, 4], seed=16)
    x = pw.arrays()
    t = Dev(x)
    o = canary((8, pw.HV, pw.DV), pw.out_dtype)
    with pytest.raises(TypeError):
        gdn.gdn_prefill(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"],
                        t["cu_seqlens"].to(torch.int64), o)
    with pytest.raises(ValueError):
        gdn.gdn_prefill(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"],
                        t["indices"][:1], t["cu_seqlens"], o)
    # no sequences, or no tokens: nothing enqueued, nothing written
    before = host(t["pool"])
    empty = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_prefill(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"][:0],
                    empty, o)
    torch.cuda.synchronize()
    assert np.array_equal(host(t["pool"]), before) and is_canary(host(o)).all()


@pytest.mark.parametrize("make", [W.prefill_8k, W.prefill_mix], ids=["isl8k", "mix"])
def test_prefill_full_size_sampled(make):
    """The timed workloads at full size (ISL 8K x 8 prompts; 64 prompts of 256..4096 tokens): sampled (prompt,
    head) pairs' outputs and final states against the oracle run on that (prompt, head) alone."""
    pw = make()
    x = pw.arrays()
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = run_prefill(pw, t, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_h, pool_h = host(o), host(t["pool"])
    orc = oracle.default()
    r = pw.HV // pw.HK
    rng = np.random.default_rng(2024)
    cu = x["cu_seqlens"]
    lens = np.diff(cu)
    pairs = [(0, 0), (3, pw.HV - 1), (int(lens.argmax()), 5), (int(lens.argmin()), 7)] + \
        [(int(b), int(h)) for b, h in zip(rng.integers(0, pw.B, 2), rng.integers(0, pw.HV, 2))]
    for b, h in pairs:
        lo, hi = int(cu[b]), int(cu[b + 1])
        hk = h // r
        slot = int(x["indices"][b])
        y = dict(q=np.ascontiguousarray(x["q"][lo:hi, hk:hk + 1]), k=np.ascontiguousarray(x["k"][lo:hi, hk:hk + 1]),
                 v=np.ascontiguousarray(x["v"][lo:hi, h:h + 1]), a=np.ascontiguousarray(x["a"][lo:hi, h:h + 1]),
                 b=np.ascontiguousarray(x["b"][lo:hi, h:h + 1]), A_log=np.ascontiguousarray(x["A_log"][h:h + 1]),
                 dt_bias=np.ascontiguousarray(x["dt_bias"][h:h + 1]), indices=np.zeros(1, np.int32))
        pool1 = np.ascontiguousarray(x["pool"][slot:slot + 1, h:h + 1])
        d = dict(prefill_dims(pw), HK=1, HV=1, num_slots=1)
        o_ref, fl = orc.prefill(d, y, np.array([0, hi - lo], np.int32), pool1,
                                np.array([x["has_initial_state"][b]], np.int32))
        assert fl == 0
        check_o(pw, o_h[lo:hi, h], o_ref[:, 0], f"o prompt {b} head {h}")
        check_state(pw, pool_h[slot, h], pool1[0, 0], f"state prompt {b} head {h}")


# ---- gated RMSNorm ------------------------------------------------------------------------------------------
def norm_ref(x, o_dtype, z_dtype, eps):
    return oracle.default().gated_rmsnorm(x["o"], o_dtype, x["z"], z_dtype, x["w"], eps)


def check_norm(y_gpu, ref, o_dtype, what):
    """The norm computes in fp32 (relative error ~1e-6: a sum of DV squares, one square root, expf) and rounds
    once to o's type, so: bf16 y within the rounding bound 2^-8 |ref| + 1e-4 max|ref| element-wise, with at
    least 95 % of the elements the correctly rounded value (no absolute cap: y is O(1..10), unlike the
    recurrence's outputs); fp32 y within 1e-5 max|ref|."""
    if o_dtype != "bf16":
        return assert_f32_close(y_gpu, ref, what, rel=1e-5)
    x = storage_to_f64(np.asarray(y_gpu))
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    d = np.abs(x - ref)
    bad = d > 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max()
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond the bf16 rounding bound (worst {d.max():.3e})"
    from gdn_workloads import to_bf16_bits
    exact = float((np.asarray(y_gpu) == to_bf16_bits(ref.astype(np.float32))).mean())
    assert exact >= 0.95, f"{what}: only {exact:.4f} correctly rounded"


@pytest.mark.parametrize("DV,o_dtype,z_dtype", [(128, "bf16", "bf16"), (128, "f32", "f32"), (128, "f32", "bf16"),
                                                (8, "bf16", "bf16"), (24, "bf16", "f32"), (64, "f32", "f32"),
                                                (512, "bf16", "bf16"), (100, "bf16", "bf16"), (1000, "f32", "f32"),
                                                (1, "f32", "f32"), (2048, "bf16", "bf16")])
def test_gated_rmsnorm(DV, o_dtype, z_dtype):
    rows = 1537  # ragged: not a multiple of any lane grouping
    x = W.gated_norm_inputs(rows, DV, o_dtype, z_dtype, seed=DV)
    o, z, w = dev(x["o"]), dev(x["z"]), dev(x["w"])
    y = gdn.gdn_gated_rmsnorm(o, z, w, eps=1e-6)
    torch.cuda.synchronize()
    check_norm(host(y), norm_ref(x, o_dtype, z_dtype, 1e-6), o_dtype, f"DV={DV}")


def test_gated_rmsnorm_in_place_and_misaligned():
    DV, rows = 128, 300
    x = W.gated_norm_inputs(rows, DV, "bf16", "bf16", seed=7)
    ref = norm_ref(x, "bf16", "bf16", 1e-5)
    o = dev(x["o"])
    gdn.gdn_gated_rmsnorm(o, dev(x["z"]), dev(x["w"]), o, eps=1e-5)  # in place
    torch.cuda.synchronize()
    check_norm(host(o), ref, "bf16", "in place")
    # rows starting 2 bytes off a 16-byte boundary: the column-at-a-time path
    buf_o = torch.empty(rows * DV + 1, dtype=torch.bfloat16, device="cuda")
    buf_z = torch.empty(rows * DV + 1, dtype=torch.bfloat16, device="cuda")
    buf_o[1:].copy_(dev(x["o"]).view(-1))
    buf_z[1:].copy_(dev(x["z"]).view(-1))
    y = gdn.gdn_gated_rmsnorm(buf_o[1:].view(rows, DV), buf_z[1:].view(rows, DV), dev(x["w"]), eps=1e-5)
    torch.cuda.synchronize()
    check_norm(host(y), ref, "bf16", "misaligned")


def test_gated_rmsnorm_host_checks():
    x = W.gated_norm_inputs(4, 16, "bf16", "bf16", seed=1)
    o, z, w = dev(x["o"]), dev(x["z"]), dev(x["w"])
    with pytest.raises(gdn.GdnError):
        gdn.gdn_gated_rmsnorm(o, z, w, eps=-1.0)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_gated_rmsnorm(o, z, w, eps=float("nan"))
    with pytest.raises(ValueError):
        gdn.gdn_gated_rmsnorm(o, z[:2], w)
    y = canary((0, 16), "bf16")
    gdn.gdn_gated_rmsnorm(o[:0], z[:0], w, y)  # zero rows: a no-op


def test_gated_rmsnorm_after_verify():
    """The verify step's outputs through the norm: rows = B*T*HV of DV, against the oracle's norm of the
    stored o (the call normalises what verify stored)."""
    w = W.verify_t4().replace(B=16, num_slots=32)
    x = w.arrays()
    t = Dev(x)
    o, _ = run_verify(w, t, cache=False)
    g = W.gated_norm_inputs(16 * 4 * 32, 128, "bf16", "bf16", seed=99)
    y = gdn.gdn_gated_rmsnorm(o, dev(g["z"]).view(o.shape), dev(g["w"]))
    torch.cuda.synchronize()
    o_h = host(o)
    ref = oracle.default().gated_rmsnorm(o_h.reshape(-1, 128), "bf16", g["z"], "bf16", g["w"], 1e-6)
    check_norm(host(y).reshape(-1, 128), ref, "bf16", "norm after verify")
