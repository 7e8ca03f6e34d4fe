"""Host logic of bench.py, on the CPU: algorithmic byte counts, per-rank workloads, the max/sum over ranks
with two gloo ranks, and the reference arm (the oracle) end to end on the tiny workload."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import gdn_workloads as W


def test_algorithmic_bytes_verify_t4():
    w = W.verify_t4()
    # state read 128*32*16384*2 + cache write 4x that + per token q,k (2*16*128*2), v, o (32*128*2 each), a, b
    state = 128 * 32 * 128 * 128 * 2
    per_tok = 2 * 16 * 128 * 2 + 2 * 32 * 128 * 2 + 2 * 32 * 2
    assert bench.recurrent_bytes(w, 128) == state + 4 * state + 128 * 4 * per_tok + 32 * 8 + 128 * 4
    assert bench.commit_bytes(w, 128) == 2 * state + 2 * 128 * 4


def test_algorithmic_bytes_replay_and_decode():
    w = W.verify_t4_replay()
    state = 128 * 32 * 128 * 128 * 2
    per_tok = 2 * 16 * 128 * 2 + 2 * 32 * 128 * 2 + 2 * 32 * 2
    assert bench.recurrent_bytes(w, 128) == state + 128 * 4 * per_tok + 32 * 8 + 128 * 4
    in_tok = 2 * 16 * 128 * 2 + 32 * 128 * 2 + 2 * 32 * 2
    assert bench.commit_bytes(w, 128, 300) == 2 * state + 2 * 128 * 4 + 300 * in_tok + 32 * 8
    d = W.decode_t1()
    fstate = 64 * 32 * 128 * 128 * 4
    assert bench.recurrent_bytes(d, 64) == 2 * fstate + 64 * (2 * 16 * 128 * 2 + 2 * 32 * 128 * 2 + 2 * 32 * 2) \
        + 32 * 8 + 64 * 4


def test_kernel_names_follow_the_launcher_rule():
    sms = 152
    v4, v8, d1 = W.verify_t4(), W.verify_t8(), W.decode_t1()
    assert bench.kernel_name(v4, "verify", sms) == "gdn_recurrent_staged_kernel"  # bf16, T=4: 8 bytes per row elt
    assert bench.kernel_name(v4, "commit", sms) == "gdn_commit_kernel"
    assert bench.kernel_name(v8, "verify", sms) == "gdn_recurrent_kernel"  # T * 2 bytes > 8
    r4 = W.verify_t4_replay()
    assert bench.kernel_name(r4, "verify", sms) == "gdn_verify_chunked_kernel"  # no cache, bf16 pool, T <= 8
    assert bench.kernel_name(r4, "commit_replay", sms) == "gdn_verify_chunked_kernel"
    assert bench.kernel_name(d1, "decode", sms) in ("gdn_recurrent_staged_kernel", "gdn_recurrent_kernel")
    assert bench.kernel_name(W.tiny(), "verify", sms) == "gdn_recurrent_kernel"  # a handful of CTAs: never staged


def test_e2e_inputs_pack_and_rotate_over_disjoint_slots(monkeypatch):
    """The end-to-end leg's packed host buffers hold each step input byte for byte (16-byte aligned views), and
    its slot sets keep the padding positions and are pairwise disjoint."""
    import numpy as np
    import torch

    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)  # no GPU here
    w = W.Workload("e2e_small", B=6, T=3, HK=2, HV=4, DK=32, DV=24, num_slots=40, qkv_dtype="bf16",
                   state_dtype="bf16", out_dtype="bf16", mode="verify", cache=False, commit=True, seed=5,
                   pad_fraction=0.34, commit_mode="replay")
    st = bench.Step(w, torch.device("cpu"))
    assert st.e2e_sets == 4
    idx0 = st.d["indices"].numpy()
    seen = []
    for j, hb in enumerate(st.h_sets):
        st.dev_slots[1].copy_(hb)
        v = st.slot_views[1]
        for k in st.step_keys:
            assert v[k].data_ptr() % 16 == 0 and v[k].shape == st.d[k].shape and v[k].dtype == st.d[k].dtype
            if k != "indices":
                assert torch.equal(v[k].view(torch.uint8), st.d[k].view(torch.uint8)), k
        idx = v["indices"].numpy()
        assert np.array_equal(idx < 0, idx0 < 0)
        if j == 0:
            assert np.array_equal(idx, idx0)
        act = set(idx[idx >= 0].tolist())
        assert len(act) == int((idx >= 0).sum()) and max(act) < w.num_slots
        assert all(not (act & other) for other in seen)
        seen.append(act)
    assert st.h2d_bytes == sum(st.d[k].numel() * st.d[k].element_size() for k in st.step_keys)


def test_rank_workloads_differ_only_in_seed():
    w = W.verify_t4()
    w1 = bench.rank_workload(w, 1)
    assert bench.rank_workload(w, 0) is w
    assert w1.seed != w.seed and w1.replace(seed=w.seed) == w


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    dist = bench.init_dist(world, "gloo")
    mx = bench.max_over_ranks(10.0 + rank, dist)
    sm = bench.sum_over_ranks(1.0 + rank, dist)
    q.put((rank, mx, sm))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 11.0, 3.0), (1, 11.0, 3.0)]


def test_reference_arm_tiny():
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3",
                           "--ref-seconds", "2"]) == 0
    j = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "tokens/s"
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["cpu_baseline"]["kind"] == "oracle"
    assert j["config"]["workload"] == W.tiny().name


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"]) == 0
    assert buf.getvalue() == ""


def test_prefill_and_norm_reference_arms_small():
    """The oracle arms of the prefill and gated-norm lines, on small inputs: one JSON line each, the oracle as
    the reference, nothing copied."""
    import argparse

    args = argparse.Namespace(steps=3, warmup=3, ref_seconds=1.0)
    pw = W.PrefillWorkload("prefill_small", B=3, HK=2, HV=4, DK=16, DV=16, num_slots=5, qkv_dtype="bf16",
                           state_dtype="bf16", out_dtype="bf16", seed=9, lengths=(20, 0, 7), pad_fraction=0.0)
    for run, unit, name in ((lambda: bench.run_prefill_reference_arm(args, pw, 0, 1), "tokens/s", pw.name),
                            (lambda: bench.run_norm_reference_arm(args, 0, 1, rows=512, DV=64), "rows/s",
                             "gated_rmsnorm_rows512_DV64_bf16")):
        buf = io.StringIO()
        with redirect_stdout(buf):
            run()
        j = json.loads(buf.getvalue().strip().splitlines()[-1])
        assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == unit
        assert j["config"]["workload"] == name and j["cpu_baseline"]["kind"] == "oracle"
        assert j["e2e"]["h2d_bytes_per_step"] == 0
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_prefill_reference_arm(args, pw, 1, 2)  # other ranks do no work
    assert buf.getvalue() == ""


def test_prefill_cpu_baseline_small():
    pw = W.PrefillWorkload("prefill_small", B=2, HK=1, HV=2, DK=16, DV=16, num_slots=4, qkv_dtype="f32",
                           state_dtype="f32", out_dtype="f32", seed=10, lengths=(5, 9))
    cb = bench._prefill_cpu_baseline(pw, pw.arrays(), 0.05)
    assert cb["value"] > 0 and cb["kind"] == "oracle" and cb["cores"] == bench.host_cores()
    assert cb["one_thread"]["value"] > 0 and cb["cpu_model"]


def test_alu_peak_derivation():
    assert abs(bench.alu_peak_tflops(152, 2070) - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9


def test_cpu_baseline_uses_every_core_and_reports_one_thread():
    cb = bench.cpu_baseline(W.tiny(), 0.3)
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_cores() >= 1
    assert cb["value"] > 0 and cb["one_thread"]["value"] > 0 and cb["one_thread"]["pairs"] >= 1
    assert cb["cpu_model"] and str(cb["cores"]) in cb["sample"]


def test_oracle_throughput_runs_items_in_order_until_done_or_deadline():
    import threading

    seen, lock = [], threading.Lock()

    def item(i):
        def f():
            with lock:
                seen.append(i)
        return f

    n, dt = bench.oracle_throughput([item(i) for i in range(50)], 1e9, 4)
    assert n == 50 and sorted(seen) == list(range(50)) and dt >= 0
    n, _ = bench.oracle_throughput([item(i) for i in range(50)], -1.0, 4)  # deadline already passed
    assert n == 0


def test_clock_summary_takes_the_median_under_load():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.max_mhz, cs.source, cs.period = 2070, "test", 0.01
    # (sm MHz, W, reason bits, utilisation %): two idle samples at a low clock, three busy ones
    cs.samples = [(900, 100.0, 0x1, 0), (2070, 900.0, 0, 100), (2000, 950.0, 0x4, 100), (2070, 910.0, 0, 90),
                  (900, 100.0, 0x1, 0)]
    s = cs.summary()
    assert s["sm_mhz"] == 2070 and s["samples"] == 5 and s["samples_under_load"] == 3 and s["sm_mhz_min"] == 2000
    assert s["reasons"] == ["sw_power_cap"]  # gpu_idle is not a throttle reason


def test_roofline_block_reports_both_peaks():
    k = {"kernel": "k", "role": "verify", "achieved_gbs": 6400.0, "frac": 6400.0 / 6790.0, "algorithmic_bytes": 1,
         "avg_us": 1.0}
    r = bench.roofline_block(k, 6790.0, "measured (x)", None)
    assert abs(r["frac"] - 6400 / 6790) < 1e-12 and abs(r["frac_nominal"] - 0.8) < 1e-12
    assert r["nominal_peak"] == 8000.0 and r["peak"] == 6790.0 and "of measured" in r["peak_source"]


def test_fused_step_bytes_and_kernel():
    w = W.verify_t4_fused()
    state = 128 * 32 * 128 * 128 * 2
    per_tok = 2 * 16 * 128 * 2 + 2 * 32 * 128 * 2 + 2 * 32 * 2
    prev_tok = 16 * 128 * 2 + 32 * 128 * 2 + 2 * 32 * 2
    assert bench.fused_bytes(w, 128, 300) == 2 * state + 128 * 4 * per_tok + 300 * prev_tok + 32 * 8 + 2 * 128 * 4
    assert bench.kernel_name(w, "verify_commit", 152) == "gdn_verify_chunked_kernel"
    assert bench.kernel_name(w.replace(state_dtype="f32"), "verify_commit", 152).count("gdn_recurrent_kernel") == 2
    p = W.previous_step(w)
    assert p["k"].shape == (128, 4, 16, 128) and p["accept_len"].min() >= 1 and p["accept_len"].max() <= 4
    assert not (p["k"] == w.small_arrays()["k"]).all()  # its own draws


def test_prefill_roofline_counts():
    """The chunked prefill's MMA flops and algorithmic bytes, recomputed by hand on two sequences (40 and 0 tokens
    of an active lane, 33 tokens of a padded one): two chunks of one item per head for the first, none for the
    others; bytes of the 40 tokens and one state written and read (it has an initial state)."""
    import bench
    pw = W.PrefillWorkload("t", B=3, HK=1, HV=2, DK=128, DV=128, num_slots=4, qkv_dtype="bf16", state_dtype="bf16",
                           out_dtype="bf16", seed=1, lengths=(40, 0, 33), fresh_fraction=0.0)
    x = pw.small_arrays()
    x["indices"] = np.array([2, 0, -1], np.int32)
    per_chunk = 2 * 2 * 128 * 64 * 128 + 2 * 128 * 64 * 128 + 3 * 2 * 128 * 32 * 32 + 2 * 2 * 128 * 128 * 32
    assert bench.prefill_mma_flops(pw, x) == per_chunk * 2 * 2
    per_tok = (2 * 128 + 2 * 128 + 2 * 2) * 2 + 2 * 128 * 2
    assert bench.prefill_bytes(pw, x) == 40 * per_tok + 2 * (2 * 128 * 128 * 2)
    assert bench.prefill_mma_flops(pw.replace(qkv_dtype="f32"), x) is None  # the other token path: not counted
    assert not bench.prefill_is_chunked(pw.replace(DK=256))


def test_in_proj_counts():
    """The in_proj line's algorithmic bytes and flops, recomputed by hand: W once, the active rows' x and outputs,
    the state read (and written back, or the records), taps and bias, indices; 2 x rows x C x H flops plus the
    convolution's 2 K per convolved output."""
    import bench
    w = W.InProjWorkload("t", B=3, T=2, H=64, HK=1, HV=2, DK=16, DV=8, K=4, num_slots=5, conv_dtype="bf16",
                         out_dtype="f32", seed=1)
    Cc, C = 2 * 16 + 2 * 8, 2 * 16 + 2 * 8 + 2 * 8 + 2 * 2
    assert (w.Cc, w.C) == (Cc, C)
    rows = 2 * 2  # two active lanes
    common = C * 64 * 2 + rows * 64 * 2 + rows * C * 4 + 2 * 3 * Cc * 2 + Cc * 5 * 4 + 3 * 4
    assert bench.in_proj_counts(w, 2, decode=True) == (common + 2 * 3 * Cc * 2, 2 * rows * C * 64 + 2 * 4 * rows * Cc)
    assert bench.in_proj_counts(w, 2, decode=False)[0] == common + rows * Cc * 2


def test_in_proj_reference_arm_small(monkeypatch):
    """The oracle arm of an in_proj line on a small projection: one JSON line, the oracle as the reference."""
    import argparse

    small = W.InProjWorkload("in_proj_small", B=3, T=2, H=64, HK=1, HV=2, DK=16, DV=8, K=4, num_slots=5,
                             conv_dtype="bf16", out_dtype="bf16", seed=2)
    monkeypatch.setitem(bench.IN_PROJ_NAMED, "in_proj16", lambda: small)
    args = argparse.Namespace(steps=3, warmup=3, ref_seconds=1.0)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_in_proj_reference_arm(args, "in_proj16", 0, 1)
    j = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "rows/s"
    assert j["config"]["workload"] == "in_proj_small" and j["cpu_baseline"]["kind"] == "oracle"
    assert j["e2e"]["h2d_bytes_per_step"] == 0
