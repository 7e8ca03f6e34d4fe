"""gdn_mtp_verify_gated, gdn_decode_gated (and the norm of gdn_mtp_verify_commit) on the GPU: o and the pool exactly
as the calls without the norm leave them, and y = the gated RMSNorm of that stored o.

o is checked against the oracle's verify as usual; y against the oracle's gated norm of the o the GPU stored
(the call's definition: the norm of the stored o), with the norm's tolerance.  Three ways to the norm are covered:
inside the chunked verify kernel (bf16 pool, no intermediate states, T <= 8, DK >= 64, DV <= 128), as the epilogue
of the token-by-token kernels (every other verify, and decode: the CTAs of one head run as one thread-block cluster
of at most 8 and meet through distributed shared memory; clusters of 1, 3, 4 and 7 CTAs, direct and staged kernels),
and the standalone norm launch after the kernel (a head wider than 8 CTAs, or a grid of more than one wave).  Rows of padded lanes must be left
untouched in y."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gated_deltanet_linear_mtp_gb300 as gdn
import gdn_workloads as W
import oracle
from gpu_util import Dev, canary, check_o, dev, host, is_canary
from test_gpu_parity import compare_verify
from test_gpu_prefill import check_norm


def wl(name, B=6, T=4, HK=2, HV=4, DK=128, DV=128, state="bf16", qkv="bf16", out="bf16", seed=80, pad=0.2):
    return W.Workload(name, B=B, T=T, HK=HK, HV=HV, DK=DK, DV=DV, num_slots=13, qkv_dtype=qkv, state_dtype=state,
                      out_dtype=out, mode="verify", cache=False, commit=False, seed=seed, pool_std=0.1,
                      pad_fraction=pad)


def gate_inputs(w, z_dtype, seed):
    g = W.gated_norm_inputs(w.B * w.T * w.HV, w.DV, w.out_dtype, z_dtype, seed=seed)
    z = g["z"].reshape(w.B, w.T, w.HV, w.DV)
    return z, g["w"]


def check_y(w, x, o_h, y_h, z, wt, eps, z_dtype):
    act = x["indices"] >= 0
    assert is_canary(y_h[~act]).all(), "y of a padded lane was written"
    if act.any():
        ref = oracle.default().gated_rmsnorm(np.ascontiguousarray(o_h[act]), w.out_dtype, np.ascontiguousarray(z[act]),
                                             z_dtype, wt, eps)
        check_norm(y_h[act], ref, w.out_dtype, "y")


CASES = [
    # fused: the norm inside the chunked verify kernel
    (wl("gv_fused_T4"), "bf16", False),
    (wl("gv_fused_T8_zf32", T=8, seed=81), "f32", False),
    (wl("gv_fused_dv96_T3", DV=96, T=3, seed=82), "bf16", False),
    (wl("gv_fused_f32out", qkv="f32", out="f32", seed=83), "f32", False),
    (wl("gv_fused_dk64_T1", DK=64, T=1, seed=84), "bf16", False),
    # the token-by-token kernels with the norm as their epilogue: a cache, DV > 128, an fp32 pool, DK < 64, T > 8
    (wl("gv_cache_T4", seed=85), "bf16", True),
    (wl("gv_dv200", DV=200, seed=86), "bf16", False),
    (wl("gv_f32state", state="f32", out="f32", qkv="f32", seed=87), "f32", False),
    (wl("gv_dk32", DK=32, DV=48, seed=88), "bf16", False),
    (wl("gv_T12", T=12, DV=64, seed=89), "bf16", False),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w,z_dtype,cache", CASES, ids=lambda c: c.name if isinstance(c, W.Workload) else str(c))
def test_verify_gated(w, z_dtype, cache):
    x = w.arrays()
    z, wt = gate_inputs(w, z_dtype, seed=w.seed + 7)
    t = Dev(x)
    o = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    y = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    c = canary((w.B, w.T, w.HV, w.DV, w.DK), w.state_dtype) if cache else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_mtp_verify_gated(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"],
                             o, gdn.GatedNorm(dev(z), dev(wt), y, eps=1e-6), c, err, scale=w.scale, l2_eps=w.l2_eps)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_h, y_h = host(o), host(y)
    compare_verify(w, x, o_h, host(c) if cache else None)
    check_y(w, x, o_h, y_h, z, wt, 1e-6, z_dtype)
    # o is exactly what gdn_mtp_verify writes
    o2 = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    gdn.gdn_mtp_verify(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"], o2,
                       canary((w.B, w.T, w.HV, w.DV, w.DK), w.state_dtype) if cache else None,
                       scale=w.scale, l2_eps=w.l2_eps)
    torch.cuda.synchronize()
    b1 = o_h.view(np.uint32) if o_h.dtype == np.float32 else o_h
    o2h = host(o2)
    b2 = o2h.view(np.uint32) if o2h.dtype == np.float32 else o2h
    assert np.array_equal(b1, b2), "o differs from gdn_mtp_verify's"


@pytest.mark.gpu
def test_verify_gated_in_place():
    """y = o: o is replaced by its gated norm."""
    w = wl("gv_in_place", seed=90)
    x = w.arrays()
    z, wt = gate_inputs(w, "bf16", seed=97)
    t = Dev(x)
    o = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    o_ref = canary((w.B, w.T, w.HV, w.DV), w.out_dtype)
    gdn.gdn_mtp_verify(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"],
                       o_ref, None)
    gdn.gdn_mtp_verify_gated(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"],
                             o, gdn.GatedNorm(dev(z), dev(wt), o, eps=1e-6))
    torch.cuda.synchronize()
    check_y(w, x, host(o_ref), host(o), z, wt, 1e-6, "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("T,Tp", [(4, 3), (8, 2)])
def test_verify_commit_with_the_norm(T, Tp):
    """The one-pass step (T, T' <= 4) and the two-launch step (T = 8) with the gated norm: o and the pool exactly
    as without the norm, y the norm of that o."""
    w = wl(f"gv_commit_T{T}_Tp{Tp}", T=T, seed=91 + T)
    x = w.arrays()
    xp = w.replace(T=Tp, seed=w.seed + 50).small_arrays()
    z, wt = gate_inputs(w, "bf16", seed=w.seed + 9)
    rt = {k: dev(xp[k]) for k in ("k", "v", "a", "b", "accept_len")}
    prev = gdn.ReplayTokens(rt["k"], rt["v"], rt["a"], rt["b"], rt["accept_len"])
    outs = []
    for with_norm in (True, False):
        t = Dev(x)
        o = canary((w.B, T, w.HV, w.DV), w.out_dtype)
        y = canary((w.B, T, w.HV, w.DV), w.out_dtype)
        norm = gdn.GatedNorm(dev(z), dev(wt), y, eps=1e-6) if with_norm else None
        gdn.gdn_mtp_verify_commit(prev, t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"],
                                  t["indices"], o, norm=norm)
        torch.cuda.synchronize()
        outs.append((host(o), host(t["pool"]), host(y)))
    (o1, p1, y1), (o2, p2, _) = outs
    assert np.array_equal(o1, o2) and np.array_equal(p1, p2), "the norm changed o or the pool"
    check_y(w, x, o1, y1, z, wt, 1e-6, "bf16")


def dwl(name, B, HV, HK=2, DK=128, DV=128, state="bf16", qkv="bf16", out="bf16", seed=120, pad=0.2):
    return W.Workload(name, B=B, T=1, HK=HK, HV=HV, DK=DK, DV=DV, num_slots=B + 5, qkv_dtype=qkv, state_dtype=state,
                      out_dtype=out, mode="decode", cache=False, commit=False, seed=seed, pool_std=0.1,
                      pad_fraction=pad)


DECODE_CASES = [
    # staged kernel, a whole head per CTA (a cluster of one): bf16 pool, 384 CTAs
    (dwl("dg_staged_head", B=12, HV=32, HK=16), "bf16"),
    # direct kernel (few CTAs): 4 CTAs of 32 rows per head, one cluster of 4
    (dwl("dg_direct_c4", B=3, HV=4, seed=121), "f32"),
    # fp32 pool, staged 16 KiB: 32 rows per CTA, clusters of 4 (512 CTAs: one wave)
    (dwl("dg_f32_staged", B=4, HV=32, HK=16, state="f32", out="f32", qkv="f32", seed=122), "f32"),
    # clusters of 3 and 7; DK = 32 (128 rows per CTA: a cluster of one in the direct kernel)
    (dwl("dg_dv96", B=3, HV=4, DV=96, seed=123), "bf16"),
    (dwl("dg_dv200", B=2, HV=2, HK=1, DV=200, seed=124), "bf16"),
    (dwl("dg_dk32", B=4, HV=4, DK=32, DV=64, seed=125), "bf16"),
    # the norm's own launch after the decode: a head of 10 CTAs (wider than one cluster), and a grid of 2048 CTAs
    # (more than one wave)
    (dwl("dg_dv300_fallback", B=2, HV=2, HK=1, DV=300, seed=126), "bf16"),
    (dwl("dg_waves_fallback", B=64, HV=32, HK=16, seed=128), "bf16"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w,z_dtype", DECODE_CASES, ids=lambda c: c.name if isinstance(c, W.Workload) else str(c))
def test_decode_gated(w, z_dtype):
    """gdn_decode_gated: o and the written-back pool bit for bit as gdn_decode leaves them, y the gated norm of that
    stored o (the oracle's, at the norm's tolerance), rows of padded lanes untouched."""
    x = w.arrays()
    z, wt = gate_inputs(w, z_dtype, seed=w.seed + 7)
    outs = []
    for gated in (True, False):
        t = Dev(x)
        o = canary((w.B, 1, w.HV, w.DV), w.out_dtype)
        y = canary((w.B, 1, w.HV, w.DV), w.out_dtype)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if gated:
            gdn.gdn_decode_gated(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"],
                                 t["indices"], o, gdn.GatedNorm(dev(z), dev(wt), y, eps=1e-6), err, scale=w.scale,
                                 l2_eps=w.l2_eps)
        else:
            gdn.gdn_decode(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"],
                           o, err, scale=w.scale, l2_eps=w.l2_eps)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((host(o), host(t["pool"]), host(y)))
    (o1, p1, y1), (o2, p2, _) = outs
    bits = lambda a: a.view(np.uint32) if a.dtype == np.float32 else a  # noqa: E731  (padded rows hold NaN canaries)
    assert np.array_equal(bits(o1), bits(o2)) and np.array_equal(bits(p1), bits(p2)), "the norm changed o or the pool"
    check_y(w, x, o1, y1, z, wt, 1e-6, z_dtype)


@pytest.mark.gpu
@pytest.mark.parametrize("state", ["bf16", "f32"])
def test_decode_gated_in_place(state):
    """y = o: each CTA reads its rows' o from its own shared memory before writing y over them."""
    w = dwl(f"dg_in_place_{state}", B=3, HV=4, state=state, out=state, qkv=state, seed=127)
    x = w.arrays()
    z, wt = gate_inputs(w, "bf16", seed=131)
    t = Dev(x)
    o_ref = canary((w.B, 1, w.HV, w.DV), w.out_dtype)
    gdn.gdn_decode(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], Dev(x)["pool"], t["indices"],
                   o_ref)
    o = canary((w.B, 1, w.HV, w.DV), w.out_dtype)
    gdn.gdn_decode_gated(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"], t["indices"],
                         o, gdn.GatedNorm(dev(z), dev(wt), o, eps=1e-6))
    torch.cuda.synchronize()
    check_y(w, x, host(o_ref), host(o), z, wt, 1e-6, "bf16")


@pytest.mark.gpu
def test_decode_gated_graph_capture():
    """The fused decode norm (a thread-block-cluster launch) captured into a CUDA graph before any eager call of its
    shape, then replayed: o, y and the written-back pool as eager calls leave them, step after step."""
    w = dwl("dg_graph", B=3, HV=4, seed=129)
    x = w.arrays()
    z, wt = gate_inputs(w, "bf16", seed=132)
    t, te = Dev(x), Dev(x)
    shape = (w.B, 1, w.HV, w.DV)
    o, y, oe, ye = (canary(shape, w.out_dtype) for _ in range(4))
    zd, wd = dev(z), dev(wt)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gdn.gdn_decode_gated(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["pool"],
                             t["indices"], o, gdn.GatedNorm(zd, wd, y))
    for rep in range(3):
        g.replay()
        gdn.gdn_decode_gated(te["q"], te["k"], te["v"], te["a"], te["b"], te["A_log"], te["dt_bias"], te["pool"],
                             te["indices"], oe, gdn.GatedNorm(zd, wd, ye))
        torch.cuda.synchronize()
        for a, b_, what in ((o, oe, "o"), (y, ye, "y"), (t["pool"], te["pool"], "pool")):
            ha, hb = host(a), host(b_)
            if ha.dtype == np.float32:
                ha, hb = ha.view(np.uint32), hb.view(np.uint32)
            assert np.array_equal(ha, hb), (rep, what)
