"""gdn_in_proj_conv and gdn_conv_commit on the GPU against the CPU oracle, through the C ABI.

The cases aim at what the kernel adds:
* the tile edges: channel counts that leave the last 128-channel tile ragged, hidden sizes that leave the last
  64-column chunk ragged, more than 64 rows (several row tiles, the last ragged), lanes gathered ahead in shared
  memory with aligned and unaligned state rows;
* the split of the hidden dimension over a cluster (every small case runs 2..8 ranks; one chunk runs alone);
* every tap count (2, 3, 4), T from 1 to 16, bf16 and fp32 state and outputs, SiLU on and off;
* padded lanes (untouched, bit for bit), a bad index (flag bit), the decode write-back and the verify's records;
* the commit of the records, bit for bit, and verify + commit against decode of the accepted rows;
* the three timed workloads at full size (hidden 2048, 12352 channels);
* two host threads on their own streams (the per-device tiling cache shared), and a new shape captured into a
  CUDA graph and replayed.

Tolerances (the kernel accumulates in fp32 on the tensor cores, the oracle in fp64):
* the stored pre-convolution values (records, the written-back state): 1 ulp of the state type as in
  ``gpu_util`` (bf16: at most 1 ulp where the two sums straddle a rounding midpoint; fp32: 1e-4 of the maximum);
* z, b, a: the fp32 / bf16 output rules of ``gpu_util``;
* q, k, v (after the convolution): those rules plus, for a bf16 state, 1.1 * sum_j |w_j| ulp(seq_j): the largest
  change a 1-ulp difference of every stored input could make through the taps and the SiLU (slope <= 1.1).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gated_deltanet_linear_mtp_gb300 as gdn
import gdn_workloads as W
import oracle
from gpu_util import (assert_bf16_stored_close, assert_f32_close, bf16_ulp, canary, dev, host, is_canary,
                      storage_to_f64)

pytestmark = pytest.mark.gpu


def small(name, B=3, T=4, H=256, HK=2, HV=4, DK=32, DV=32, K=4, conv="bf16", out="bf16", silu=True, seed=600,
          pad=0.0, num_slots=None):
    return W.InProjWorkload(name, B=B, T=T, H=H, HK=HK, HV=HV, DK=DK, DV=DV, K=K, num_slots=num_slots or B + 3,
                            conv_dtype=conv, out_dtype=out, seed=seed, silu=silu, pad_fraction=pad)


def odims(w):
    return dict(T=w.T, H=w.H, HK=w.HK, HV=w.HV, DK=w.DK, DV=w.DV, K=w.K, num_slots=w.num_slots, x_dtype="bf16",
                conv_dtype=w.conv_dtype, silu=int(w.silu))


def outputs(w):
    B, T = w.B, w.T
    return gdn.InProjOut(canary((B, T, w.HK, w.DK), w.out_dtype), canary((B, T, w.HK, w.DK), w.out_dtype),
                         canary((B, T, w.HV, w.DV), w.out_dtype), canary((B, T, w.HV, w.DV), w.out_dtype),
                         canary((B, T, w.HV), w.out_dtype), canary((B, T, w.HV), w.out_dtype))


def run_gpu(w, x, write_state, records=True, err=None, indices=None):
    t = {k: dev(v) for k, v in x.items()}
    if indices is not None:
        t["indices"] = dev(indices)
    out = outputs(w)
    rec = canary((w.B, w.T, w.Cc), w.conv_dtype) if records else None
    gdn.gdn_in_proj_conv(t["x"], t["W"], t["conv_w"], t["conv_b"], t["conv_state"], t["indices"], out, write_state,
                         rec, err, silu=w.silu)
    torch.cuda.synchronize()
    got = {n: host(getattr(out, n)) for n in ("q", "k", "v", "z", "b", "a")}
    return got, (host(rec) if records else None), host(t["conv_state"])


def gpu_flat(w, got):
    """The outputs [B, T, C] in channel order (as fp64)."""
    B, T = w.B, w.T
    return np.concatenate([storage_to_f64(got[n]).reshape(B, T, -1) for n in ("q", "k", "v", "z", "b", "a")], axis=-1)


def conv_slack(w, x, pool_before, rec_ref, idx):
    """Per element of the convolved channels: 1.1 * sum_j |w_j| * ulp(seq_j) for a bf16 state, else 0."""
    B, T, K, Cc = w.B, w.T, w.K, w.Cc
    if w.conv_dtype != "bf16":
        return np.zeros((B, T, Cc))
    taps = np.abs(x["conv_w"].astype(np.float64))  # [Cc, K]
    out = np.zeros((B, T, Cc))
    for b in range(B):
        if idx[b] < 0:
            continue
        seq = np.concatenate([storage_to_f64(pool_before[idx[b]]), storage_to_f64(rec_ref[b])], axis=0)  # [K-1+T, Cc]
        u = bf16_ulp(seq)
        for t in range(T):
            out[b, t] = 1.1 * (taps * u[t:t + K].T).sum(axis=1)
    return out


def compare_outputs(w, x, got, ref_out, rec_ref, pool_before, idx):
    act = idx >= 0
    Cc = w.Cc
    for n in ("q", "k", "v", "z", "b", "a"):
        assert is_canary(got[n][~act]).all(), f"{n} of a padded lane was written"
    if not act.any():
        return
    g = gpu_flat(w, got)[act]
    r = ref_out[act]
    slack = conv_slack(w, x, pool_before, rec_ref, idx)[act]
    scale = np.abs(r).max()
    d = np.abs(g - r)
    if w.out_dtype == "bf16":
        bound = 2.0 ** -8 * np.abs(r) + 1e-4 * scale
    else:
        bound = np.full(r.shape, 1e-4 * scale)
    bound[..., :Cc] += slack
    bad = d > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outputs beyond the bound; worst at "
                           f"{np.unravel_index(np.argmax(d - bound), d.shape)}: {d.max():.3e}")
    assert d[..., Cc:].max() <= (2e-2 if w.out_dtype == "bf16" else 1e-4 * scale)


def compare_stored(w, got, ref, what):
    if w.conv_dtype == "bf16":
        assert_bf16_stored_close(got, ref, what, min_exact=0.9)
    else:
        assert_f32_close(got, ref, what)


def check_call(w, x, write_state):
    idx = x["indices"]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got, rec, pool = run_gpu(w, x, write_state, records=not write_state, err=err)
    assert int(err.item()) == 0
    pool_ref = x["conv_state"].copy()
    ref_out, rec_ref, flags = oracle.default().in_proj_conv(odims(w), x["x"], x["W"], x["conv_w"], x["conv_b"],
                                                            pool_ref, idx, write_pool=write_state, records=True)
    assert flags == 0
    compare_outputs(w, x, got, ref_out, rec_ref, x["conv_state"], idx)
    act = idx >= 0
    untouched = np.setdiff1d(np.arange(w.num_slots), idx[act])
    if write_state:
        assert np.array_equal(pool[untouched], x["conv_state"][untouched]), "a slot no lane uses was written"
        compare_stored(w, pool[idx[act]], pool_ref[idx[act]], "state")
    else:
        assert np.array_equal(pool, x["conv_state"]), "verify rows wrote the state"
        assert is_canary(rec[~act]).all(), "records of a padded lane were written"
        compare_stored(w, rec[act], rec_ref[act], "records")


SMALL = [
    small("ip_bf16_T4"),
    small("ip_f32_T2", T=2, conv="f32", out="f32", seed=601),
    small("ip_ragged_H_K3_nosilu_pad", B=5, T=1, H=200, K=3, silu=False, conv="bf16", out="f32", pad=0.4, seed=602),
    small("ip_K2_T8_one_chunk", B=2, T=8, H=64, K=2, conv="f32", out="bf16", seed=603),
    small("ip_T16", B=2, T=16, H=128, HK=1, HV=2, DK=64, DV=48, seed=604),
    small("ip_wide_heads", B=2, T=3, H=512, HK=2, HV=6, DK=128, DV=96, seed=605),
    # 160 rows (64-row tiles, lanes gathered ahead in shared memory) with 9 convolved channels: rows not 16-byte
    # aligned, so the state comes by direct loads
    small("ip_odd_channels_gathered", B=40, T=4, H=64, HK=1, HV=1, DK=3, DV=3, seed=608, pad=0.25),
    # 48 rows: two tiles of 24 rows (6 lanes), ragged 16-row padding
    small("ip_two_tiles_48_rows", B=12, T=4, H=128, seed=609, pad=0.2),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("write_state", [True, False], ids=["decode", "verify"])
def test_small(w, write_state):
    check_call(w, w.arrays(), write_state)


@pytest.mark.parametrize("write_state", [True, False], ids=["decode", "verify"])
def test_two_row_tiles(write_state):
    """320 rows: five tiles of 16 lanes x 4 rows (the lanes gathered ahead), a tile of only non-convolved channels."""
    w = small("ip_rows320", B=80, T=4, H=128, HK=1, HV=2, DK=32, DV=32, pad=0.1, seed=606, num_slots=90)
    check_call(w, w.arrays(), write_state)


def test_bad_index():
    w = small("ip_bad_index", B=4, seed=607)
    x = w.arrays()
    idx = x["indices"].copy()
    idx[2] = w.num_slots
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got, _, pool = run_gpu(w, x, True, records=False, err=err, indices=idx)
    assert int(err.item()) == gdn.ERRBIT_INDEX
    for n in got:
        assert is_canary(got[n][2]).all()
    assert np.array_equal(pool[np.setdiff1d(np.arange(w.num_slots), idx[[0, 1, 3]])],
                          x["conv_state"][np.setdiff1d(np.arange(w.num_slots), idx[[0, 1, 3]])])


@pytest.mark.parametrize("conv,K", [("bf16", 4), ("f32", 3), ("bf16", 2)])
def test_conv_commit(conv, K):
    """Bit for bit against the oracle's commit of the same records: L in 0..T, a padded lane, a bad length and a bad
    index (their slots untouched, flag bits set)."""
    w = small(f"cc_{conv}_K{K}", B=6, T=4, K=K, conv=conv, seed=610 + K)
    x = w.arrays()
    idx = x["indices"].copy()
    L = np.array([0, 1, 2, 4, 3, 5], np.int32)     # lane 5: L > T
    idx[4] = -1
    t_state, t_idx, t_rec, t_L = dev(x["conv_state"]), dev(idx), dev(x["records"]), dev(L)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_conv_commit(t_state, t_idx, t_rec, t_L, err)
    torch.cuda.synchronize()
    ref = x["conv_state"].copy()
    flags = oracle.default().conv_commit(odims(w), ref, idx, x["records"], L)
    assert flags == 2 and int(err.item()) == gdn.ERRBIT_ACCEPT_LEN
    assert np.array_equal(host(t_state), ref)
    idx[1] = w.num_slots + 3
    err.zero_()
    gdn.gdn_conv_commit(t_state, dev(idx), t_rec, t_L, err)
    torch.cuda.synchronize()
    assert int(err.item()) & gdn.ERRBIT_INDEX


def test_verify_then_commit_is_decode_of_the_accepted_rows():
    """The state after verify rows + the commit of L of them equals the oracle's decode of those L rows."""
    w = small("ip_chain", B=4, T=4, seed=620)
    x = w.arrays()
    L = np.array([1, 4, 2, 3], np.int32)
    t = {k: dev(v) for k, v in x.items()}
    rec = canary((w.B, w.T, w.Cc), w.conv_dtype)
    gdn.gdn_in_proj_conv(t["x"], t["W"], t["conv_w"], t["conv_b"], t["conv_state"], t["indices"], outputs(w), False,
                         rec)
    gdn.gdn_conv_commit(t["conv_state"], t["indices"], rec, dev(L))
    torch.cuda.synchronize()
    pool = host(t["conv_state"])
    orc = oracle.default()
    for b in range(w.B):
        wl = w.replace(B=1, T=int(L[b]))
        ref = x["conv_state"].copy()
        orc.in_proj_conv(odims(wl), np.ascontiguousarray(x["x"][b:b + 1, :L[b]]), x["W"], x["conv_w"], x["conv_b"],
                         ref, x["indices"][b:b + 1], write_pool=True, records=False)
        s = x["indices"][b]
        compare_stored(w, pool[s], ref[s], f"lane {b}")


@pytest.mark.parametrize("make,write_state", [(W.in_proj_verify16, False), (W.in_proj_decode8, True)],
                         ids=["verify16", "decode8"])
def test_full_size(make, write_state):
    """The timed workloads: every lane, every channel."""
    w = make()
    check_call(w, w.arrays(), write_state)


def test_full_size_512_rows_sampled():
    """The 512-row verify (eight row tiles of 16 lanes): lanes from several tiles and their edges against the oracle
    run on those lanes alone."""
    w = W.in_proj_verify512()
    x = w.arrays()
    got, rec, pool = run_gpu(w, x, False)
    assert np.array_equal(pool, x["conv_state"])
    lanes = np.array([0, 63, 64, 127, 17, 100])
    xs = dict(x, x=np.ascontiguousarray(x["x"][lanes]), indices=np.ascontiguousarray(x["indices"][lanes]))
    ws = w.replace(B=len(lanes))
    ref_out, rec_ref, _ = oracle.default().in_proj_conv(odims(ws), xs["x"], x["W"], x["conv_w"], x["conv_b"],
                                                        x["conv_state"].copy(), xs["indices"], write_pool=False)
    compare_outputs(ws, xs, {n: v[lanes] for n, v in got.items()}, ref_out, rec_ref, x["conv_state"], xs["indices"])
    compare_stored(ws, rec[lanes], rec_ref, "records")


def _eager(w, x, t, write_state, stream=None):
    out = outputs(w)
    rec = None if write_state else canary((w.B, w.T, w.Cc), w.conv_dtype)
    gdn.gdn_in_proj_conv(t["x"], t["W"], t["conv_w"], t["conv_b"], t["conv_state"], t["indices"], out, write_state,
                         rec, silu=w.silu, stream=stream)
    return out, rec


def test_calls_from_two_host_threads():
    """Two host threads on their own streams call the kernel over and over with different shapes (different splits:
    the per-device tiling cache is shared and overwritten by both); every result equals the single-threaded one bit
    for bit (the split-K sum is formed in rank order, so it is deterministic)."""
    import threading

    cases = [small("thr_a", B=4, T=4, H=512, seed=630), small("thr_b", B=3, T=2, H=384, HK=2, HV=6, DK=64, DV=48,
                                                              seed=631)]
    prepared = []
    for w in cases:
        x = w.arrays()
        t = {k: dev(v) for k, v in x.items()}
        out, rec = _eager(w, x, t, False)
        torch.cuda.synchronize()
        prepared.append((w, x, t, {n: host(getattr(out, n)) for n in ("q", "k", "v", "z", "b", "a")}, host(rec)))
    failures = []

    def worker(w, x, t, ref, rec_ref):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for _ in range(30):
                    out, rec = _eager(w, x, t, False, stream=stream)
                stream.synchronize()
                for n, r in ref.items():
                    if not np.array_equal(host(getattr(out, n)), r):
                        failures.append(f"{w.name}: {n} differs")
                if not np.array_equal(host(rec), rec_ref):
                    failures.append(f"{w.name}: records differ")
        except Exception as e:  # surfaced below
            failures.append(f"{w.name}: {e!r}")

    threads = [threading.Thread(target=worker, args=a) for a in prepared]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not failures, failures


def test_graph_capture_of_a_new_shape():
    """A shape never launched before is captured into a CUDA graph (its split is chosen during the capture) and
    replayed: decode rows move the state on at every replay, as eager calls do."""
    w = small("graph_new_shape", B=5, T=1, H=320, HK=3, HV=6, DK=32, DV=40, seed=640)
    x = w.arrays()
    t = {k: dev(v) for k, v in x.items()}
    te = {k: dev(v) for k, v in x.items()}  # eager twin
    out = outputs(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gdn.gdn_in_proj_conv(t["x"], t["W"], t["conv_w"], t["conv_b"], t["conv_state"], t["indices"], out, True,
                             None, silu=w.silu)
    for rep in range(3):
        g.replay()
        oe, _ = _eager(w, x, te, True)
        torch.cuda.synchronize()
        for n in ("q", "k", "v", "z", "b", "a"):
            assert np.array_equal(host(getattr(out, n)), host(getattr(oe, n))), (rep, n)
        assert np.array_equal(host(t["conv_state"]), host(te["conv_state"])), rep
    # and the first replay's outputs are the oracle's decode from the initial state
    check_call(w, x, True)
