"""gdn_mtp_verify_commit on the GPU: one speculative step that commits the accepted prefix of an earlier call and
verifies this call's tokens from the committed states.

Checked against the oracle as the composition the call defines: the oracle's replay commit of the earlier tokens
into a copy of the pool, then the oracle's verify of the new tokens from that pool.  The result must also equal,
bit for bit, the two separate GPU calls gdn_commit_replay + gdn_mtp_verify: on the one-pass path (bf16 pool, both
token counts <= 4, DK >= 64) by the same arithmetic with the committed rows read from the tile instead of the
pool, and outside it because the call runs those two calls itself."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import gated_deltanet_linear_mtp_gb300 as gdn
import gdn_workloads as W
import oracle
from gpu_util import Dev, canary, check_o, check_state, dev, host, is_canary, storage_to_f64

pytestmark = pytest.mark.gpu

LANE_KEYS = ("q", "k", "v", "a", "b", "indices", "accept_len")


def step_inputs(w: W.Workload, Tp: int, seed_prev: int, zero_frac: float = 0.0):
    """Inputs of one step (the workload's T tokens and pool) and of the earlier call on the same lanes (Tp tokens,
    its own draws, accept lengths U{1..Tp}, a fraction of them set to 0)."""
    x = w.arrays()
    xp = w.replace(T=Tp, seed=seed_prev).small_arrays()
    xp["indices"] = x["indices"]
    acc = xp["accept_len"].copy()
    rng = np.random.default_rng([seed_prev, 7])
    acc[rng.random(w.B) < zero_frac] = 0
    xp["accept_len"] = acc
    xp["A_log"], xp["dt_bias"] = x["A_log"], x["dt_bias"]
    return x, xp


def take(x: dict, lanes) -> dict:
    y = dict(x)
    for k in LANE_KEYS:
        if k in x:
            y[k] = np.ascontiguousarray(x[k][lanes])
    return y


def oracle_step(w, Tp, x, xp, lanes=None, chunk=16):
    """(o [lanes, T, HV, DV] fp64, pool after the step) from the oracle: replay commit of xp's accepted tokens into
    a copy of the pool, then verify of x's tokens from it; lanes in chunks on a few threads."""
    orc = oracle.default()
    d_new, d_prev = oracle.dims_of(w), dict(oracle.dims_of(w), T=Tp)
    pool = x["pool"].copy()
    acc = xp["accept_len"]
    flags = orc.commit_replay(d_prev, xp, pool, acc)  # the whole batch: slots are distinct
    lanes = np.arange(w.B) if lanes is None else np.asarray(lanes)

    def part(i):
        xs = take(dict(x, pool=pool), lanes[i:i + chunk])
        o, _, _ = orc.verify(d_new, xs, cache=False)
        return o

    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        o = np.concatenate(list(ex.map(part, range(0, len(lanes), chunk))), axis=0)
    return o, pool, flags


def run_step(w, x, xp, err=None, stream=None):
    t = Dev(x)
    tp = {k: dev(xp[k]) for k in ("k", "v", "a", "b", "accept_len")}
    o = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    gdn.gdn_mtp_verify_commit(gdn.ReplayTokens(tp["k"], tp["v"], tp["a"], tp["b"], tp["accept_len"]), t["q"], t["k"],
                              t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"], o, err,
                              scale=w.scale, l2_eps=w.l2_eps, stream=stream)
    return o, t, tp


def run_two_calls(w, x, xp, t, tp):
    """gdn_commit_replay of the earlier tokens into a copy of the original pool, then gdn_mtp_verify."""
    pool = dev(x["pool"])
    qp = tp["k"]  # q of the earlier call is not read for outputs
    gdn.gdn_commit_replay(qp, tp["k"], tp["v"], tp["a"], tp["b"], t["A_log"], t["dt_bias"], pool, t["indices"],
                          tp["accept_len"], scale=w.scale, l2_eps=w.l2_eps)
    o = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    gdn.gdn_mtp_verify(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], pool, t["indices"], o, None,
                       scale=w.scale, l2_eps=w.l2_eps)
    return o, pool


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def oracle_verify_from(w, x, pool, lanes, chunk=16):
    """The oracle's verify of x's tokens from a given pool (the one the GPU committed)."""
    orc = oracle.default()

    def part(i):
        o, _, _ = orc.verify(oracle.dims_of(w), take(dict(x, pool=pool), lanes[i:i + chunk]), cache=False)
        return o

    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        return np.concatenate(list(ex.map(part, range(0, len(lanes), chunk))), axis=0)


def check_step(w, Tp, x, xp, o_gpu, pool_gpu, lanes=None):
    """The committed slots against the oracle's replay commit (the stored-bf16 tolerance: a state rounded from
    fp32 may differ from the one rounded from fp64 by one ulp); o against the oracle's verify from the pool as the
    GPU committed it (the o tolerance), and against the oracle's whole step within the 2e-2 max-abs of o."""
    o_ref, pool_ref, flags = oracle_step(w, Tp, x, xp, lanes)
    idx, acc = x["indices"], xp["accept_len"]
    lanes = np.arange(w.B) if lanes is None else np.asarray(lanes)
    act = idx[lanes] >= 0
    og = o_gpu[lanes]
    if act.any():
        o_own = oracle_verify_from(w, x, pool_gpu, lanes)
        check_o(w, og[act], o_own[act], "o (from the committed state)")
        d = np.abs(storage_to_f64(og[act]) - o_ref[act]).max()
        assert d <= 2e-2, f"o: max-abs {d:.3e} from the oracle's whole step"
    assert is_canary(og[~act]).all(), "o of a padded lane was written"
    committed = (idx >= 0) & (acc >= 1) & (acc <= Tp)
    sl = idx[committed]
    if len(sl):
        check_state(w, pool_gpu[sl], pool_ref[sl], "committed slots")
    untouched = np.setdiff1d(np.arange(w.num_slots), sl)
    assert np.array_equal(pool_gpu[untouched], x["pool"][untouched]), "a slot without a commit changed"
    return flags


def small(name, B=5, T=3, HK=2, HV=4, DK=64, DV=40, num_slots=11, state="bf16", qkv="bf16", out="bf16", seed=40,
          pad=0.2):
    return W.Workload(name, B=B, T=T, HK=HK, HV=HV, DK=DK, DV=DV, num_slots=num_slots, qkv_dtype=qkv,
                      state_dtype=state, out_dtype=out, mode="verify", cache=False, commit=True, seed=seed,
                      pool_std=0.1, pad_fraction=pad)


# the one-pass kernel takes a bf16 pool, DK >= 64 and both token counts <= 4; the other cases run the two calls
CASES = [
    (small("vc_dk64_dv40_T3_Tp2"), 2, 0.2),
    (small("vc_dk128_dv200_T4_Tp4", DK=128, DV=200, B=6, T=4, seed=41), 4, 0.3),
    (small("vc_dk128_T8_Tp1", DK=128, DV=128, T=8, seed=42), 1, 0.0),
    (small("vc_dk128_T1_Tp8", DK=128, DV=128, T=1, seed=43), 8, 0.0),
    (small("vc_dk256_dv64_T2_Tp5", DK=256, DV=64, T=2, seed=44), 5, 0.2),
    (small("vc_f32in_dk128_T3_Tp3", DK=128, DV=96, qkv="f32", out="f32", seed=45), 3, 0.2),
    (small("vc_hv_8x_hk", HK=1, HV=8, DK=128, DV=128, T=4, seed=46), 3, 0.0),
    (small("vc_f32state_T2_Tp3", state="f32", out="f32", qkv="f32", seed=47), 3, 0.2),
    (small("vc_dk32_bf16", DK=32, DV=33, seed=48), 2, 0.2),
    (small("vc_T12_Tp3", DK=128, DV=64, T=12, seed=49), 3, 0.0),
    (small("vc_T4_Tp10", DK=128, DV=64, T=4, seed=50), 10, 0.0),
]


@pytest.mark.parametrize("w,Tp,zero", CASES, ids=lambda c: c.name if isinstance(c, W.Workload) else str(c))
def test_verify_commit_against_the_oracle_and_the_two_calls(w, Tp, zero):
    x, xp = step_inputs(w, Tp, seed_prev=w.seed + 1000, zero_frac=zero)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, t, tp = run_step(w, x, xp, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_h, pool_h = host(o), host(t["pool"])
    check_step(w, Tp, x, xp, o_h, pool_h)
    o2, pool2 = run_two_calls(w, x, xp, t, tp)
    torch.cuda.synchronize()
    # bit patterns: the padded lanes hold NaN canaries
    assert np.array_equal(bits(host(o2)), bits(o_h)), "o differs from gdn_commit_replay + gdn_mtp_verify"
    assert np.array_equal(bits(host(pool2)), bits(pool_h)), "the pool differs from gdn_commit_replay + gdn_mtp_verify"


@pytest.mark.parametrize("w", [W.verify_t4(), W.verify_t8()], ids=lambda w: w.name)
def test_verify_commit_full_size(w):
    """The T=4 (B=128) and T=8 (B=256, 26 padded lanes) verify workloads, each committing an earlier call of its
    own width first: every lane's o and every slot against the oracle."""
    w = w.replace(cache=False)
    x, xp = step_inputs(w, w.T, seed_prev=w.seed + 500, zero_frac=0.05)
    o, t, tp = run_step(w, x, xp)
    torch.cuda.synchronize()
    check_step(w, w.T, x, xp, host(o), host(t["pool"]))


def test_bad_accept_lengths_commit_nothing_and_set_the_bit():
    w = small("vc_bad_len", DK=128, DV=128, B=6, T=4, seed=51, pad=0.0)
    x, xp = step_inputs(w, 4, seed_prev=52)
    xp["accept_len"][1] = 5   # beyond the earlier call's 4 tokens
    xp["accept_len"][3] = -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, t, _ = run_step(w, x, xp, err)
    torch.cuda.synchronize()
    assert int(err.item()) & gdn.ERRBIT_ACCEPT_LEN
    xr = dict(xp)
    xr["accept_len"] = np.where((xp["accept_len"] < 0) | (xp["accept_len"] > 4), 0, xp["accept_len"]).astype(np.int32)
    check_step(w, 4, x, xr, host(o), host(t["pool"]))


def test_width_transitions_as_one_pass_steps():
    """Six steps on one pool, widths 8, 1, 3, 2, 8, 4: each step commits the previous step's accepted prefix and
    verifies its own tokens in one call (the first commits nothing); every step's o and the pool against an oracle
    that runs the same chain from its own pool."""
    widths = (8, 1, 3, 2, 8, 4)
    base = small("vc_chain", B=7, HK=2, HV=4, DK=128, DV=128, num_slots=16, seed=60, pad=0.15)
    orc = oracle.default()
    first = base.replace(T=1).arrays()
    pool_ref, idx = first["pool"], first["indices"]
    pool_gpu = dev(pool_ref)
    prev = None
    for i, T in enumerate(widths):
        w = base.replace(T=T, seed=61 + i)
        x = w.small_arrays()
        x["pool"] = pool_ref
        if prev is None:  # nothing to commit yet: an earlier call of width 1 with accept lengths 0
            xp = w.replace(T=1, seed=99).small_arrays()
            xp["accept_len"] = np.zeros(w.B, np.int32)
        else:
            xp = prev
        xp["indices"] = x["indices"] = idx
        Tp = xp["k"].shape[1]
        t = Dev(x)
        tp = {k: dev(xp[k]) for k in ("k", "v", "a", "b", "accept_len")}
        o = canary((w.B, T, w.HV, w.DV), w.out_dtype)
        gdn.gdn_mtp_verify_commit(gdn.ReplayTokens(tp["k"], tp["v"], tp["a"], tp["b"], tp["accept_len"]), t["q"],
                                  t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], pool_gpu, t["indices"], o)
        torch.cuda.synchronize()
        xq = dict(xp, A_log=x["A_log"], dt_bias=x["dt_bias"])
        ph = host(pool_gpu)
        check_step(w, Tp, x, xq, host(o), ph)
        pool_ref = ph  # the next step starts from the pool the GPU left
        prev = w.small_arrays()
        prev["A_log"], prev["dt_bias"] = x["A_log"], x["dt_bias"]
        prev["accept_len"] = np.random.default_rng([70, i]).integers(0, T + 1, size=w.B).astype(np.int32)
