"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on the same seeded inputs.

Full-size checks use the workloads the benchmark times (decode T=1 B=64 fp32 state; verify T=4 B=128 bf16
state + commit; verify T=8 B=256 with 10 % padded lanes), plus the B x T x dtype sweep on sampled lanes and
small edge cases that span several row tiles with a ragged tail.  Tolerances: see ``gpu_util``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import gated_deltanet_linear_mtp_gb300 as gdn
import gdn_workloads as W
import oracle
from gpu_util import (Dev, assert_bf16_stored_close, assert_f32_close, canary, check_o, check_state, dev, host,
                      is_canary, run_decode, run_verify, storage_to_f64)

pytestmark = pytest.mark.gpu

LANE_KEYS = ("q", "k", "v", "a", "b", "indices", "accept_len")


def take_lanes(x: dict, lanes) -> dict:
    lanes = np.asarray(lanes)
    y = dict(x)
    for k in LANE_KEYS:
        y[k] = np.ascontiguousarray(x[k][lanes])
    return y


def compare_verify(w, x, o_gpu, cache_gpu, lanes=None, chunk=16):
    """o / cache of the given lanes against the oracle; padded and invalid lanes must hold canaries.  The
    oracle runs on chunks of lanes in a few threads (its calls release the GIL), at most a few chunks ahead
    of the comparison."""
    orc = oracle.default()
    d = oracle.dims_of(w)
    B = x["q"].shape[0]
    lanes = np.arange(B) if lanes is None else np.asarray(lanes)
    starts = list(range(0, len(lanes), chunk))

    def ref(i):
        xs = take_lanes(x, lanes[i:i + chunk])
        return xs, orc.verify(d, xs, cache=cache_gpu is not None)

    workers = max(1, min(8, (os.cpu_count() or 1)))
    with ThreadPoolExecutor(workers) as ex:
        futs = {}
        for j, i in enumerate(starts):
            for i2 in starts[j:j + workers]:
                if i2 not in futs:
                    futs[i2] = ex.submit(ref, i2)
            xs, (o_ref, c_ref, _) = futs.pop(i).result()
            _check_chunk(w, xs, lanes[i:i + chunk], o_gpu, cache_gpu, o_ref, c_ref)


def _check_chunk(w, xs, sel, o_gpu, cache_gpu, o_ref, c_ref):
    act = (xs["indices"] >= 0) & (xs["indices"] < w.num_slots)
    og = o_gpu[sel]
    if act.any():
        check_o(w, og[act], o_ref[act], f"o lanes {sel[act][:4]}..")
    if (~act).any():
        assert is_canary(og[~act]).all(), "o of a skipped lane was written"
    if cache_gpu is not None:
        cg = cache_gpu[sel]
        if act.any():
            check_state(w, cg[act], c_ref[act], f"cache lanes {sel[act][:4]}..")
        if (~act).any():
            assert is_canary(cg[~act]).all(), "cache of a skipped lane was written"


def check_commit(w, x, pool_before_gpu, pool_after, cache_gpu):
    """Committed slots equal cache[b, L-1] bit for bit; every other slot is unchanged bit for bit."""
    idx, acc = x["indices"], x["accept_len"]
    touched = np.zeros(w.num_slots, bool)
    for b in range(len(idx)):
        s = idx[b]
        if 0 <= s < w.num_slots and 1 <= acc[b] <= w.T:
            assert np.array_equal(pool_after[s], cache_gpu[b, acc[b] - 1]), f"lane {b}"
            touched[s] = True
    assert np.array_equal(pool_after[~touched], pool_before_gpu[~touched]), "an uncommitted slot changed"


def pool_host_pair(t):
    return host(t["pool"])


# ---------------------------------------------------------------------------------------------------------
def test_tiny_verify_commit_decode():
    w = W.tiny()
    x = w.arrays()
    t = Dev(x)
    o, cache = run_verify(w, t, cache=True)
    torch.cuda.synchronize()
    o_h, c_h = host(o), host(cache)
    compare_verify(w, x, o_h, c_h)
    # commit
    before = host(t["pool"])
    gdn.gdn_commit(t["pool"], t["indices"], cache, t["accept_len"])
    after = host(t["pool"])
    check_commit(w, x, before, after, c_h)
    # decode of the same tokens one at a time from the original pool == the cached states
    pool = dev(x["pool"])
    w1 = w.replace(T=1, mode="decode")
    for tok in range(w.T):
        xt = dict(x)
        for k in ("q", "k", "v", "a", "b"):
            xt[k] = np.ascontiguousarray(x[k][:, tok:tok + 1])
        ot = run_decode(w1, Dev(xt), pool)
        ph = host(pool)
        for b, s in enumerate(x["indices"]):
            assert_f32_close(ph[s], c_h[b, tok], f"decode step {tok} lane {b}")
        assert_f32_close(host(ot)[:, 0], o_h[:, tok], f"decode o step {tok}")


def test_decode_t1_full():
    w = W.decode_t1()
    x = w.arrays()
    t = Dev(x)
    pool_before = host(t["pool"])
    o = run_decode(w, t, t["pool"])
    torch.cuda.synchronize()
    o_h, pool_gpu = host(o), host(t["pool"])
    orc = oracle.default()
    pool_ref = x["pool"].copy()
    o_ref, fl = orc.decode(oracle.dims_of(w), x, pool_ref)
    assert fl == 0
    check_o(w, o_h, o_ref)
    idx = x["indices"]
    check_state(w, pool_gpu[idx], pool_ref[idx], "pool write-back")
    untouched = np.setdiff1d(np.arange(w.num_slots), idx)
    assert np.array_equal(pool_gpu[untouched], pool_before[untouched])


def test_verify_t4_full_and_commit():
    w = W.verify_t4()
    x = w.arrays()
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, cache = run_verify(w, t, cache=True, err=err)
    torch.cuda.synchronize()
    pool_before = host(t["pool"])
    assert np.array_equal(pool_before, x["pool"]), "verify wrote the pool"
    o_h, c_h = host(o), host(cache)
    compare_verify(w, x, o_h, c_h)
    gdn.gdn_commit(t["pool"], t["indices"], cache, t["accept_len"], err)
    check_commit(w, x, pool_before, host(t["pool"]), c_h)
    assert int(err.item()) == 0


def test_verify_t8_padded_every_lane_and_commit():
    """Full-size verify T=8 (B=256, 26 padded lanes): o and every cached state of all 230 active lanes against
    the oracle, every padded lane untouched, then the commit bit for bit."""
    w = W.verify_t8()
    x = w.arrays()
    idx = x["indices"]
    assert (idx == -1).sum() == 26
    t = Dev(x)
    o, cache = run_verify(w, t, cache=True)
    torch.cuda.synchronize()
    o_h, c_h = host(o), host(cache)
    compare_verify(w, x, o_h, c_h)
    # every padded lane untouched, everywhere
    assert is_canary(o_h[idx < 0]).all() and is_canary(c_h[idx < 0]).all()
    pool_before = host(t["pool"])
    gdn.gdn_commit(t["pool"], t["indices"], cache, t["accept_len"])
    check_commit(w, x, pool_before, host(t["pool"]), c_h)


# ---- the sweep, on sampled lanes ---------------------------------------------------------------------
_POOLS = {}


def _sweep_pool(w):
    key = (w.state_dtype, w.pool_seed)
    if key not in _POOLS:
        p = w.pool()
        _POOLS.clear()
        _POOLS[key] = (p, dev(p))
    return _POOLS[key]


@pytest.mark.parametrize("w", W.sweep(), ids=lambda w: w.name)
def test_sweep_point(w):
    x = w.small_arrays()
    pool_h, pool_d = _sweep_pool(w)
    x["pool"] = pool_h
    t = Dev({k: v for k, v in x.items() if k != "pool"})
    t.t["pool"] = pool_d
    lanes = np.arange(w.B) if w.B <= 8 else np.sort(np.random.default_rng(w.seed).choice(w.B, 8, replace=False))
    if w.mode == "decode":
        pool = pool_d.clone()
        o = run_decode(w, t, pool)
        torch.cuda.synchronize()
        orc = oracle.default()
        xs = take_lanes(x, lanes)
        pool_ref = pool_h.copy()
        o_ref, _ = orc.decode(oracle.dims_of(w), xs, pool_ref)
        check_o(w, host(o)[lanes], o_ref)
        sl = xs["indices"]
        check_state(w, host(pool[torch.from_numpy(sl).long().cuda()]), pool_ref[sl], "pool write-back")
        del pool
    else:
        o, cache = run_verify(w, t, cache=True)
        torch.cuda.synchronize()
        o_h, c_h = host(o), host(cache)
        compare_verify(w, x, o_h, c_h, lanes=lanes)
        pool = pool_d.clone()
        gdn.gdn_commit(pool, t["indices"], cache, t["accept_len"])
        torch.cuda.synchronize()
        sl = x["indices"]
        after = host(pool[torch.from_numpy(sl).long().cuda()])
        for j, b in enumerate(range(w.B)):
            assert np.array_equal(after[j], c_h[b, x["accept_len"][b] - 1])
        del pool, cache


# ---- edge cases: several row tiles, ragged tails, every DK, dtype mixes -----------------------------
def verify_is_chunked(w) -> bool:
    """Verify without intermediate states on a bf16 pool with T <= 8 and DK >= 64 runs the chunked tensor-core
    kernel."""
    return w.state_dtype == "bf16" and w.T <= 8 and w.DK >= 64


def small(name, B=3, T=3, HK=2, HV=4, DK=64, DV=40, num_slots=7, qkv="bf16", state="bf16", out="bf16",
          seed=0, scale=1.0, pad=0.0):
    return W.Workload(name, B=B, T=T, HK=HK, HV=HV, DK=DK, DV=DV, num_slots=num_slots, qkv_dtype=qkv,
                      state_dtype=state, out_dtype=out, mode="verify", cache=True, commit=True, seed=seed,
                      pool_std=0.1, scale=scale, pad_fraction=pad)


EDGE = [
    small("dk16_dv16_f32_all", DK=16, DV=16, qkv="f32", state="f32", out="f32"),
    small("dk16_dv200_ragged", DK=16, DV=200),
    small("dk32_dv33_f32state", DK=32, DV=33, state="f32"),
    small("dk64_dv40_ragged", DK=64, DV=40),
    small("dk128_dv100_ragged_T16", DK=128, DV=100, T=16),
    small("dk128_dv128_T1", DK=128, DV=128, T=1),
    small("dk256_dv24_ragged", DK=256, DV=24, state="f32", out="f32"),
    small("dk256_dv64_bf16", DK=256, DV=64, T=5),
    small("hk_eq_hv", HK=4, HV=4, DK=128, DV=64),
    small("hv_8x_hk", HK=1, HV=8, DK=128, DV=48, qkv="f32"),
    small("scale_half_f32out", DK=128, DV=64, out="f32", scale=0.5),
    small("b1", B=1, DK=128, DV=128),
    small("padded_half", B=8, num_slots=12, DK=128, DV=72, pad=0.5),
    # few tokens per state byte and >= 2 CTAs per SM: the bulk-copy staged kernel (several row blocks per
    # CTA), with ragged last blocks
    small("staged_dk128_dv100_T2", B=8, HK=16, HV=48, DK=128, DV=100, T=2, num_slots=10),
    small("staged_dk64_dv200_T1", B=8, HK=16, HV=48, DK=64, DV=200, T=1, num_slots=10),
    small("staged_dk256_dv24_T2_f32", B=8, HK=16, HV=48, DK=256, DV=24, T=2, state="f32", out="f32", num_slots=10),
    small("staged_dk16_dv200_T1_f32in", B=8, HK=16, HV=48, DK=16, DV=200, T=1, qkv="f32", num_slots=10),
    small("staged_dk32_dv96_T2_f32state", B=8, HK=16, HV=48, DK=32, DV=96, T=2, state="f32", num_slots=10),
    small("staged_bf16_T4", B=8, HK=16, HV=48, DK=128, DV=136, T=4, num_slots=10),
    small("staged_padded", B=16, HK=16, HV=48, num_slots=20, DK=128, DV=136, T=2, pad=0.5),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_edge_verify(w):
    x = w.arrays()
    t = Dev(x)
    o, cache = run_verify(w, t, cache=True)
    torch.cuda.synchronize()
    compare_verify(w, x, host(o), host(cache))
    o2, _ = run_verify(w, t, cache=False)
    if verify_is_chunked(w):  # without the cache a bf16 pool with T <= 8 takes the chunked form: same tolerance
        torch.cuda.synchronize()
        compare_verify(w, x, host(o2), None)
    else:  # the same kernel without the cache gives the same o, bit for bit
        assert torch.equal(o.view(torch.int16) if o.dtype == torch.bfloat16 else o.view(torch.int32),
                           o2.view(torch.int16) if o2.dtype == torch.bfloat16 else o2.view(torch.int32))


@pytest.mark.parametrize("w", [e for e in EDGE if e.name in ("dk16_dv200_ragged", "dk128_dv100_ragged_T16",
                                                                 "dk256_dv24_ragged", "padded_half")
                               or e.name.startswith("staged")], ids=lambda w: w.name)
def test_edge_decode(w):
    w = w.replace(mode="decode")
    x = w.arrays()
    t = Dev(x)
    o = run_decode(w, t, t["pool"])
    torch.cuda.synchronize()
    pool_ref = x["pool"].copy()
    o_ref, _ = oracle.default().decode(oracle.dims_of(w), x, pool_ref)
    act = x["indices"] >= 0
    check_o(w, host(o)[act], o_ref[act])
    assert is_canary(host(o)[~act]).all()
    pg = host(t["pool"])
    check_state(w, pg[x["indices"][act]], pool_ref[x["indices"][act]], "pool")
    untouched = np.setdiff1d(np.arange(w.num_slots), x["indices"][act])
    assert np.array_equal(pg[untouched], x["pool"][untouched])


def test_all_lanes_padded_touch_nothing():
    w = small("all_pad", B=4, DK=128, DV=64)
    x = w.arrays()
    x["indices"][:] = -1
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, cache = run_verify(w, t, cache=True, err=err)
    run_decode(w, t, t["pool"], err=err, o=o)
    gdn.gdn_commit(t["pool"], t["indices"], cache, t["accept_len"], err)
    torch.cuda.synchronize()
    assert is_canary(host(o)).all() and is_canary(host(cache)).all()
    assert np.array_equal(host(t["pool"]), x["pool"])
    assert int(err.item()) == 0


def test_bad_indices_and_accept_lengths_set_error_bits():
    w = small("bad", B=6, DK=64, DV=32, num_slots=8)
    x = w.arrays()
    x["indices"][:] = [0, -1, 8, -2, 3, 5]         # 8 and -2 are out of range
    x["accept_len"][:] = [1, 1, 1, 1, 0, w.T + 1]  # lane 4: no-op; lane 5: out of range
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, cache = run_verify(w, t, cache=True, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.ERRBIT_INDEX
    oh, ch = host(o), host(cache)
    for b in (1, 2, 3):
        assert is_canary(oh[b]).all() and is_canary(ch[b]).all()
    compare_verify(w, x, oh, ch, lanes=[0, 4, 5])
    err.zero_()
    gdn.gdn_commit(t["pool"], t["indices"], cache, t["accept_len"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.ERRBIT_INDEX | gdn.ERRBIT_ACCEPT_LEN
    after = host(t["pool"])
    assert np.array_equal(after[0], ch[0, 0])
    keep = [s for s in range(8) if s != 0]
    assert np.array_equal(after[keep], x["pool"][keep])   # lanes 4 (L=0) and 5 (L>T) left slots 3, 5 alone


def test_duplicate_slots_in_verify_read_the_same_state():
    w = small("dup", B=4, DK=128, DV=64)
    x = w.arrays()
    x["indices"][:] = [2, 2, 2, 2]
    for k in ("q", "k", "v", "a", "b"):
        x[k][1:] = x[k][0]
    t = Dev(x)
    o, cache = run_verify(w, t, cache=True)
    torch.cuda.synchronize()
    oh, ch = host(o), host(cache)
    for b in (1, 2, 3):
        assert np.array_equal(oh[b], oh[0]) and np.array_equal(ch[b], ch[0])
    compare_verify(w, x, oh, ch, lanes=[0])


def test_empty_batch():
    w = small("b0", B=1)
    x = w.arrays()
    t = Dev(x)
    e = {k: v[:0] for k, v in t.t.items() if k in LANE_KEYS}
    o = torch.empty((0, w.T, w.HV, w.DV), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_mtp_verify(e["q"], e["k"], e["v"], e["a"], e["b"], t["A_log"], t["dt_bias"], t["pool"], e["indices"], o)
    torch.cuda.synchronize()


# ---- chained calls on the GPU: verify(T) == T decodes, commit(L) == L decodes ------------------------
def test_chain_verify_equals_decodes_f32():
    w = small("chain", B=5, T=6, DK=128, DV=128, num_slots=9, state="f32", out="f32")
    x = w.arrays()
    t = Dev(x)
    o, cache = run_verify(w, t, cache=True)
    pool = t["pool"].clone()
    w1 = w.replace(T=1, mode="decode")
    oh, ch = host(o), host(cache)
    for tok in range(w.T):
        xt = dict(x)
        for k in ("q", "k", "v", "a", "b"):
            xt[k] = np.ascontiguousarray(x[k][:, tok:tok + 1])
        ot = run_decode(w1, Dev(xt), pool)
        torch.cuda.synchronize()
        assert_f32_close(host(ot)[:, 0], oh[:, tok], f"o step {tok}")
        ph = host(pool)
        assert_f32_close(ph[x["indices"]], ch[:, tok], f"state step {tok}")
    # commit(L) == state after L decodes
    L = x["accept_len"]
    gdn.gdn_commit(t["pool"], t["indices"], cache, t["accept_len"])
    ref = dev(x["pool"])
    for tok in range(w.T):
        xt = dict(x)
        for k in ("q", "k", "v", "a", "b"):
            xt[k] = np.ascontiguousarray(x[k][:, tok:tok + 1])
        xt["indices"] = np.where(L > tok, x["indices"], -1).astype(np.int32)
        run_decode(w1, Dev(xt), ref)
    torch.cuda.synchronize()
    assert_f32_close(host(t["pool"])[x["indices"]], host(ref)[x["indices"]], "commit vs decodes")


# ---- streams and CUDA graphs -------------------------------------------------------------------------
def test_side_stream_and_graph_replay():
    w = small("graph", B=16, T=4, DK=128, DV=128, num_slots=32)
    x = w.arrays()
    t = Dev(x)
    pool0 = t["pool"].clone()
    o = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    cache = canary((w.B, w.T, w.HV, w.DV, w.DK), w.state_dtype)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on a side stream
        run_verify(w, t, cache=True, o=o, cache_buf=cache, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    o_eager, c_eager = host(o), host(cache)
    compare_verify(w, x, o_eager, c_eager)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_verify(w, t, cache=True, o=o, cache_buf=cache)
        gdn.gdn_commit(t["pool"], t["indices"], cache, t["accept_len"])
    rng = np.random.default_rng(3)
    for rep in range(3):
        t["pool"].copy_(pool0)
        acc = rng.integers(1, w.T + 1, w.B).astype(np.int32)
        t["accept_len"].copy_(torch.from_numpy(acc))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host(o), o_eager) and np.array_equal(host(cache), c_eager)
        xr = dict(x, accept_len=acc)
        check_commit(w, xr, host(pool0), host(t["pool"]), c_eager)


# ---- verify without intermediate states: the chunked tensor-core form for bf16 pools --------------------
NOCACHE = [small(f"nocache_dk{dk}_dv{dv}_T{T}_{qkv}", B=5, T=T, HK=2, HV=4, DK=dk, DV=dv, num_slots=9, qkv=qkv,
                 out=out, pad=0.2)
           for dk, dv, T, qkv, out in [(128, 128, 4, "bf16", "bf16"), (128, 200, 8, "bf16", "f32"),
                                       (128, 100, 1, "bf16", "bf16"), (64, 64, 3, "f32", "f32"),
                                       (256, 72, 5, "bf16", "bf16"), (32, 40, 2, "bf16", "bf16"),
                                       (16, 16, 7, "f32", "bf16"), (128, 128, 16, "bf16", "bf16")]]
# several items per CTA, key heads shared by 4 value heads, several row blocks per head, padded lanes
NOCACHE += [small("nocache_persistent_dk128_dv300_T4", B=64, T=4, HK=2, HV=8, DK=128, DV=300, num_slots=80,
                  pad=0.25),
            small("nocache_persistent_dk64_dv64_T6", B=96, T=6, HK=4, HV=16, DK=64, DV=64, num_slots=100, pad=0.1)]


@pytest.mark.parametrize("w", NOCACHE + [W.verify_t4_replay()], ids=lambda w: w.name)
def test_verify_without_cache(w):
    x = w.arrays()
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, _ = run_verify(w, t, cache=False, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oh = host(o)
    idx = x["indices"]
    act = np.flatnonzero(idx >= 0)
    lanes = act if len(act) <= 24 else np.sort(np.random.default_rng(4).choice(act, 24, replace=False))
    compare_verify(w, x, oh, None, lanes=np.concatenate([lanes, np.flatnonzero(idx < 0)]))
    # and the states it read are untouched
    assert np.array_equal(host(t["pool"]), x["pool"])


def test_chunked_bad_indices_set_error_bits():
    w = small("bad_chunked", B=6, T=4, DK=128, DV=160, num_slots=8)
    x = w.arrays()
    x["indices"][:] = [0, -1, 8, -2, 3, 5]         # 8 and -2 are out of range
    x["accept_len"][:] = [1, 1, 1, 1, 0, w.T + 1]  # lane 4: no-op; lane 5: out of range
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, _ = run_verify(w, t, cache=False, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.ERRBIT_INDEX
    oh = host(o)
    for b in (1, 2, 3):
        assert is_canary(oh[b]).all()
    compare_verify(w, x, oh, None, lanes=[0, 4, 5])
    err.zero_()
    pool = t["pool"].clone()
    run_replay(w, t, pool, t["accept_len"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.ERRBIT_INDEX | gdn.ERRBIT_ACCEPT_LEN
    after = host(pool)
    keep = [s for s in range(8) if s != 0]
    assert np.array_equal(after[keep], x["pool"][keep])  # lanes 4 (L=0) and 5 (L>T) left slots 3, 5 alone
    xs = take_lanes(x, [0])
    ref = x["pool"].copy()
    assert oracle.default().commit_replay(oracle.dims_of(w), xs, ref, xs["accept_len"]) == 0
    check_state(w, after[0], ref[0], "replayed slot 0")


def test_chunked_verify_and_replay_in_a_graph():
    """The chunked kernels' per-call host set-up (tensor map, grid) captured once and replayed."""
    w = small("graph_chunked", B=24, T=4, HK=2, HV=8, DK=128, DV=128, num_slots=40, pad=0.1)
    x = w.arrays()
    t = Dev(x)
    pool0 = t["pool"].clone()
    o = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    run_verify(w, t, cache=False, o=o)
    run_replay(w, t, t["pool"], t["accept_len"])
    torch.cuda.synchronize()
    o_eager, p_eager = host(o), host(t["pool"])
    compare_verify(w, x, o_eager, None)
    g = torch.cuda.CUDAGraph()
    t["pool"].copy_(pool0)
    with torch.cuda.graph(g):
        run_verify(w, t, cache=False, o=o)
        run_replay(w, t, t["pool"], t["accept_len"])
    for _ in range(3):
        o.copy_(canary(o.shape, w.out_dtype))
        t["pool"].copy_(pool0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host(o), o_eager) and np.array_equal(host(t["pool"]), p_eager)


def test_calls_from_two_host_threads():
    """Two host threads, each on its own stream, call verify (with and without the cache, i.e. the rank-1 and the
    chunked kernels) and the replay commit over and over; every result equals the single-threaded one bit for
    bit."""
    import threading

    cases = [small("thr_bf16", B=8, T=4, HK=2, HV=4, DK=128, DV=160, num_slots=12),
             small("thr_f32", B=6, T=3, HK=2, HV=4, DK=64, DV=72, num_slots=10, state="f32", out="f32")]
    prepared = []
    for w in cases:
        x = w.arrays()
        t = Dev(x)
        o_c, cache = run_verify(w, t, cache=True)
        o_n, _ = run_verify(w, t, cache=False)
        pool = t["pool"].clone()
        run_replay(w, t, pool, t["accept_len"])
        torch.cuda.synchronize()
        prepared.append((w, t, host(o_c), host(cache), host(o_n), host(pool)))
    failures = []

    def worker(w, t, o_c_ref, c_ref, o_n_ref, pool_ref):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for _ in range(20):
                    o_c, cache = run_verify(w, t, cache=True, stream=stream)
                    o_n, _ = run_verify(w, t, cache=False, stream=stream)
                    pool = t["pool"].clone()
                    run_replay(w, t, pool, t["accept_len"])
                stream.synchronize()
                for got, ref, what in ((host(o_c), o_c_ref, "o"), (host(cache), c_ref, "cache"),
                                       (host(o_n), o_n_ref, "o without cache"), (host(pool), pool_ref, "replay")):
                    if not np.array_equal(got, ref):
                        failures.append(f"{w.name}: {what} differs")
        except Exception as e:  # surfaced below
            failures.append(f"{w.name}: {e!r}")

    threads = [threading.Thread(target=worker, args=a) for a in prepared]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not failures, failures


# ---- replay commit: the pool state of the cached commit, without caching ------------------------------
def run_replay(w, t: Dev, pool, accept_len, err=None):
    gdn.gdn_commit_replay(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], pool, t["indices"],
                          accept_len, err, scale=w.scale, l2_eps=w.l2_eps)


def assert_replay_matches_copy(w, rep, copy, what):
    """Token-by-token replay: the cached commit's bits.  Chunked replay (bf16 pool, T <= 8): within 1 bf16 ulp
    (+1e-4 max) of them and almost all bits equal, since both round an fp32 value of the same state to bf16."""
    if verify_is_chunked(w):
        assert_bf16_stored_close(rep, copy, what, min_exact=0.97)
    else:
        assert np.array_equal(rep, copy), what


REPLAY = [W.tiny(), W.verify_t4(), W.verify_t8(), W.verify_t4_replay(), W.verify_t8_replay()] + [
    e for e in EDGE if e.name in (
        "dk16_dv200_ragged", "dk32_dv33_f32state", "dk128_dv100_ragged_T16", "dk256_dv24_ragged", "hv_8x_hk",
        "padded_half", "scale_half_f32out", "staged_dk128_dv100_T2", "staged_padded", "dk128_dv128_T1",
        "dk256_dv64_bf16")] + [w for w in NOCACHE if w.T <= 8]


@pytest.mark.parametrize("w", REPLAY, ids=lambda w: w.name)
def test_commit_replay_equals_cached_commit(w):
    x = w.arrays()
    t = Dev(x)
    _, cache = run_verify(w, t, cache=True)
    pool_copy = t["pool"].clone()
    gdn.gdn_commit(pool_copy, t["indices"], cache, t["accept_len"])
    pool_rep = t["pool"].clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_replay(w, t, pool_rep, t["accept_len"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rep = host(pool_rep)
    assert_replay_matches_copy(w, rep, host(pool_copy), "replay commit vs the cached commit")
    # and against the oracle's replay, on sampled lanes
    idx = x["indices"]
    act = np.flatnonzero(idx >= 0)
    lanes = act if len(act) <= 24 else np.sort(np.random.default_rng(9).choice(act, 24, replace=False))
    xs = take_lanes(x, lanes)
    pool_ref = x["pool"].copy()
    assert oracle.default().commit_replay(oracle.dims_of(w), xs, pool_ref, xs["accept_len"]) == 0
    sl = xs["indices"]
    check_state(w, rep[sl], pool_ref[sl], "replayed slots")
    untouched = np.setdiff1d(np.arange(w.num_slots), idx[idx >= 0])
    assert np.array_equal(rep[untouched], x["pool"][untouched])


def test_commit_replay_accept_lengths():
    w = small("replay_len", B=5, T=4, DK=128, DV=64, num_slots=9)
    x = w.arrays()
    x["accept_len"][:] = [0, w.T + 1, -1, 2, w.T]
    t = Dev(x)
    pool = t["pool"].clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_replay(w, t, pool, t["accept_len"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.ERRBIT_ACCEPT_LEN
    ph = host(pool)
    for b in (0, 1, 2):
        assert np.array_equal(ph[x["indices"][b]], x["pool"][x["indices"][b]])
    _, cache = run_verify(w, t, cache=True)
    ch = host(cache)
    for b, L in ((3, 2), (4, w.T)):
        assert_replay_matches_copy(w, ph[x["indices"][b]], ch[b, L - 1], f"lane {b}, accept_len {L}")


# ---- seeded random shapes through every call ---------------------------------------------------------------
def _random_case(i):
    r = np.random.default_rng([77, i])
    DK = int(r.choice([16, 32, 64, 128, 256]))
    HK = int(r.integers(1, 4))
    HV = HK * int(r.integers(1, 5))
    T = int(r.choice([1, 2, 3, 4, 5, 7, 8, 12, 16]))
    B = int(r.integers(1, 12))
    state = str(r.choice(["bf16", "f32"]))
    qkv = str(r.choice(["bf16", "f32"]))
    out = str(r.choice(["bf16", "f32"]))
    DV = int(r.integers(1, 300))
    return small(f"random{i}_dk{DK}_dv{DV}_h{HK}x{HV}_T{T}_B{B}_{state}", B=B, T=T, HK=HK, HV=HV, DK=DK, DV=DV,
                 num_slots=B + int(r.integers(0, 6)), qkv=qkv, state=state, out=out, seed=100 + i,
                 pad=float(r.choice([0.0, 0.3])))


@pytest.mark.parametrize("i", range(24))
def test_random_shapes_every_call(i):
    """verify with and without the cache (the rank-1 and, for bf16 T <= 8, the chunked kernels), the copy and
    the replay commits, and decode, on one seeded random shape, against the oracle."""
    w = _random_case(i)
    x = w.arrays()
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, cache = run_verify(w, t, cache=True, err=err)
    o2, _ = run_verify(w, t, cache=False, err=err)
    pool_rep = t["pool"].clone()
    run_replay(w, t, pool_rep, t["accept_len"], err)
    pool_copy = t["pool"].clone()
    gdn.gdn_commit(pool_copy, t["indices"], cache, t["accept_len"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    compare_verify(w, x, host(o), host(cache))
    compare_verify(w, x, host(o2), None)
    check_commit(w, x, x["pool"], host(pool_copy), host(cache))
    ref = x["pool"].copy()
    assert oracle.default().commit_replay(oracle.dims_of(w), x, ref, x["accept_len"]) == 0
    check_state(w, host(pool_rep), ref, "replayed pool")
    # decode of the same shape (T tokens, written back)
    wd = w.replace(mode="decode")
    t_d = Dev(x)
    od = run_decode(wd, t_d, t_d["pool"], err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    pool_ref = x["pool"].copy()
    od_ref, _ = oracle.default().decode(oracle.dims_of(wd), x, pool_ref)
    act = (x["indices"] >= 0)
    if act.any():
        check_o(wd, host(od)[act], od_ref[act], "decode o")
        sl = x["indices"][act]
        check_state(wd, host(t_d["pool"])[sl], pool_ref[sl], "decode write-back")


# ---- degenerate cases of the method and maximum sizes ------------------------------------------------------
def _degenerate_case(kind, state="f32", qkv="f32", out="f32"):
    w = small(f"degenerate_{kind}", B=2, T=4, HK=1, HV=2, DK=128, DV=64, num_slots=4, qkv=qkv, state=state, out=out)
    x = w.arrays()
    rng = np.random.default_rng(8)
    as_store = (lambda a: np.asarray(a, np.float32)) if qkv == "f32" else W.to_bf16_bits
    if kind == "orthonormal":  # g = 1, beta = 1, keys orthonormal, q = k: the delta rule writes v exactly
        Q, _ = np.linalg.qr(rng.standard_normal((128, 128)))
        keys = Q[:, :w.T].T.astype(np.float32)
        k = np.broadcast_to(keys[None, :, None, :], x["k"].shape).copy()
        x["k"] = as_store(k)
        x["q"] = as_store(k)
        x["a"] = as_store(np.full(x["a"].shape, -np.inf, np.float32))
        x["b"] = as_store(np.full(x["b"].shape, np.inf, np.float32))
    elif kind == "beta0":  # beta = 0: pure decay
        x["b"] = as_store(np.full(x["b"].shape, -np.inf, np.float32))
    elif kind == "zero_keys":  # k = 0: kh = 0, no write, pure decay
        x["k"] = as_store(np.zeros(x["k"].shape, np.float32))
    return w, x


@pytest.mark.parametrize("kind", ["orthonormal", "beta0", "zero_keys"])
@pytest.mark.parametrize("state", ["f32", "bf16"])
def test_degenerate_cases(kind, state):
    w, x = _degenerate_case(kind, state=state, qkv="f32" if state == "f32" else "bf16",
                            out="f32" if state == "f32" else "bf16")
    t = Dev(x)
    o, cache = run_verify(w, t, cache=True)
    torch.cuda.synchronize()
    oh, ch = host(o), host(cache)
    assert np.all(np.isfinite(storage_to_f64(oh))) and np.all(np.isfinite(storage_to_f64(ch)))
    compare_verify(w, x, oh, ch)
    if kind == "orthonormal" and state == "f32":
        v = storage_to_f64(x["v"])
        assert np.abs(storage_to_f64(oh) - v).max() <= 1e-5 * np.abs(v).max() + 1e-6
    if verify_is_chunked(w):  # the chunked forms of verify and of the replay commit on the same inputs
        o2, _ = run_verify(w, t, cache=False)
        pool = t["pool"].clone()
        run_replay(w, t, pool, t["accept_len"])
        torch.cuda.synchronize()
        assert np.all(np.isfinite(storage_to_f64(host(o2))))
        compare_verify(w, x, host(o2), None)
        ref = x["pool"].copy()
        assert oracle.default().commit_replay(oracle.dims_of(w), x, ref, x["accept_len"]) == 0
        check_state(w, host(pool), ref, "replayed pool")


def test_maximum_batch():
    """B = 65535 lanes (the grid's z limit), tiny heads; sampled lanes against the oracle."""
    w = W.Workload("max_B", B=65535, T=2, HK=1, HV=1, DK=16, DV=16, num_slots=65535, qkv_dtype="bf16",
                   state_dtype="bf16", out_dtype="bf16", mode="verify", cache=True, commit=True, seed=11,
                   pool_std=0.1, pad_fraction=0.05)
    x = w.arrays()
    t = Dev(x)
    o, cache = run_verify(w, t, cache=True)
    torch.cuda.synchronize()
    oh, ch = host(o), host(cache)
    lanes = np.sort(np.random.default_rng(3).choice(w.B, 48, replace=False))
    lanes = np.unique(np.concatenate([lanes, [0, w.B - 1]]))
    compare_verify(w, x, oh, ch, lanes=lanes)
    pool_before = host(t["pool"])
    gdn.gdn_commit(t["pool"], t["indices"], cache, t["accept_len"])
    check_commit(w, x, pool_before, host(t["pool"]), ch)


def test_maximum_batch_chunked():
    """B = 65535 lanes through the chunked verify and replay commit: thousands of items per persistent CTA;
    sampled lanes against the oracle, every other slot untouched."""
    w = W.Workload("max_B_chunked", B=65535, T=3, HK=1, HV=2, DK=64, DV=40, num_slots=65535, qkv_dtype="bf16",
                   state_dtype="bf16", out_dtype="bf16", mode="verify", cache=False, commit=True, seed=12,
                   pool_std=0.1, pad_fraction=0.05, commit_mode="replay")
    x = w.arrays()
    t = Dev(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, _ = run_verify(w, t, cache=False, err=err)
    run_replay(w, t, t["pool"], t["accept_len"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    lanes = np.sort(np.random.default_rng(5).choice(w.B, 48, replace=False))
    lanes = np.unique(np.concatenate([lanes, [0, w.B - 1]]))
    compare_verify(w, x, host(o), None, lanes=lanes)
    after = host(t["pool"])
    xs = take_lanes(x, lanes)
    ref = x["pool"].copy()
    assert oracle.default().commit_replay(oracle.dims_of(w), xs, ref, xs["accept_len"]) == 0
    sl = xs["indices"][(xs["indices"] >= 0) & (xs["accept_len"] > 0)]
    check_state(w, after[sl], ref[sl], "replayed slots")
    idx = x["indices"]
    untouched = np.setdiff1d(np.arange(w.num_slots), idx[(idx >= 0) & (x["accept_len"] > 0)])
    assert np.array_equal(after[untouched], x["pool"][untouched])
