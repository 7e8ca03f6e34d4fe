"""Benchmark of the GDN MTP-verify step on one GB300 (or N independent replicas under torchrun).

One step = ``gdn_mtp_verify`` (T=4 draft tokens, B=128 requests, HK=16, HV=32, 128x128 bf16 states from a
512-slot pool, intermediate states cached) followed by ``gdn_commit`` of the accepted prefixes -- the MTP
verify step of sglang PR #23273 "[GDN] Enable FlashInfer MTP verify on SM100+ (Blackwell)" (NEXTN, 3 steps +
1 token; bf16 SSM state) on synthetic data.  Inputs are resident in HBM when the timed region starts;
L2 (129 MB) is flushed between steps, outside each step's CUDA events: a 256 MiB write, then a 256 MiB read
so that the lines left in L2 are clean.

    python bench.py [--steps K] [--warmup W] [--workload verify4|verify8|decode|...|sweep|sweep_replay] [--impl reference]
    python bench.py --workload prefill8k|prefill_mix|gated_norm     (the prefill and gated-norm calls, own lines)
    python bench.py --workload in_proj16|in_proj8|in_proj512        (the in_proj projection + conv1d, own lines)

Prints one JSON line (``--workload sweep``: one per point).  ``value`` = verified tokens/s (A x T per step,
A = non-padded lanes, summed over ranks, divided by the slowest rank's device time).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdn_workloads as W  # noqa: E402

METRIC = "GDN verify tokens/s and achieved HBM GB/s (% of GB300 peak) at T=1/4/8"
PREFILL_NAMED = {"prefill8k": W.prefill_8k, "prefill_mix": W.prefill_mix}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_SOURCES = ["gated_deltanet_linear_mtp_gb300/csrc/gdn_recurrent.cuh",
                  "gated_deltanet_linear_mtp_gb300/csrc/gdn_recurrent_launch.cuh",
                  "gated_deltanet_linear_mtp_gb300/csrc/gdn_verify_chunked.cuh",
                  "gated_deltanet_linear_mtp_gb300/csrc/gdn_tcgen05.cuh",
                  "gated_deltanet_linear_mtp_gb300/csrc/gdn_common.cuh",
                  "gated_deltanet_linear_mtp_gb300/csrc/gdn_commit.cu"]


def kernel_name(w, role: str, sms: int) -> str:
    """Name of the kernel the library launches for one call of the step: the rule of the launcher
    (gdn_recurrent_launch.cuh) restated for the report."""
    if role == "commit":
        return "gdn_commit_kernel"
    in_range = w.num_slots * w.HV <= 2**31 - 1 and w.B * w.HV * -(-w.DV // 128) <= 2**31 - 1
    if (w.state_dtype == "bf16" and w.T <= 8 and w.DK >= 64 and in_range
            and ((role == "verify" and not w.cache) or role in ("commit_replay", "verify_commit"))):
        return "gdn_verify_chunked_kernel"
    if role == "verify_commit":  # outside the one-pass kernel: the replay commit and the verify, two launches
        return "gdn_recurrent_kernel + gdn_recurrent_kernel"
    st = 2 if w.state_dtype == "bf16" else 4
    p = w.DK // 8
    rpc = (32 // p) * min(p, 4) * 4  # rows per CTA of the token-by-token kernels
    block = rpc * w.DK * st
    cap = (16 if (st == 4 or w.T >= 4) else 32) * 1024  # state staged per CTA
    nsub = 1 if block >= cap else min(8, cap // block)
    ctas = w.B * w.HV * -(-w.DV // (nsub * rpc))
    if w.T * st <= 8 and ctas >= 2 * sms:
        return "gdn_recurrent_staged_kernel"
    return "gdn_recurrent_kernel"


# ---------------------------------------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend)
    return dist if world > 1 else None


def max_over_ranks(x: float, dist, device=None) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist, device=None) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_workload(w: W.Workload, rank: int) -> W.Workload:
    """Weak scaling: every rank runs its own batch of the same shape (independent requests, no exchange)."""
    if rank == 0:
        return w
    return w.replace(seed=w.seed + 7919 * rank, pool_seed=None if w.pool_seed is None else w.pool_seed + 7919 * rank)


# ---- algorithmic bytes ------------------------------------------------------------------------------------
def esize(d: str) -> int:
    return 4 if d == "f32" else 2


def recurrent_bytes(w: W.Workload, A: int) -> int:
    """Bytes the method must move in one decode / verify launch for A active lanes."""
    s, i, ob = esize(w.state_dtype), esize(w.qkv_dtype), esize(w.out_dtype)
    E = w.DV * w.DK
    state_read = A * w.HV * E * s
    state_write = A * w.T * w.HV * E * s if w.cache else 0
    if w.mode == "decode":
        state_write = A * w.HV * E * s
    per_tok = 2 * w.HK * w.DK * i + w.HV * w.DV * i + w.HV * w.DV * ob + 2 * w.HV * i
    return state_read + state_write + A * w.T * per_tok + w.HV * 8 + w.B * 4


def fused_bytes(w: W.Workload, A: int, prev_accepted: int) -> int:
    """One-pass step (gdn_mtp_verify_commit): every active state read once and written once, the previous step's
    accepted tokens' k, v, a, b, and this step's q, k, v, a, b and o."""
    s, i, ob = esize(w.state_dtype), esize(w.qkv_dtype), esize(w.out_dtype)
    state = 2 * A * w.HV * w.DV * w.DK * s
    per_tok = 2 * w.HK * w.DK * i + w.HV * w.DV * i + w.HV * w.DV * ob + 2 * w.HV * i
    prev_tok = w.HK * w.DK * i + w.HV * w.DV * i + 2 * w.HV * i
    return state + A * w.T * per_tok + prev_accepted * prev_tok + w.HV * 8 + 2 * w.B * 4


def commit_bytes(w: W.Workload, A: int, accepted_tokens: int = 0) -> int:
    """Copy commit: one state read and one written per active lane.  Replay commit: the same, plus the
    accepted tokens' q, k, v, a, b (no outputs)."""
    b = 2 * A * w.HV * w.DV * w.DK * esize(w.state_dtype) + 2 * w.B * 4
    if w.commit_mode == "replay":
        i = esize(w.qkv_dtype)
        b += accepted_tokens * (2 * w.HK * w.DK * i + w.HV * w.DV * i + 2 * w.HV * i) + w.HV * 8
    return b


# ---- peaks, traffic, clocks -------------------------------------------------------------------------------
def tensor_peak():
    """Dense bf16 tensor peak for a kernel timed on its own (the burst figure)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops: cuBLAS bf16 GEMM, burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, one earlier GB300 measurement)"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


PREFILL_SOURCES = ["gated_deltanet_linear_mtp_gb300/csrc/gdn_prefill.cu",
                   "gated_deltanet_linear_mtp_gb300/csrc/gdn_prefill_chunked.cu",
                   "gated_deltanet_linear_mtp_gb300/csrc/gdn_tcgen05.cuh",
                   "gated_deltanet_linear_mtp_gb300/csrc/gdn_recurrent.cuh",
                   "gated_deltanet_linear_mtp_gb300/csrc/gdn_common.cuh"]
NORM_SOURCES = ["gated_deltanet_linear_mtp_gb300/csrc/gdn_gated_norm.cu"]


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(role: str, workload_name: str, sources=None):
    """DRAM bytes per launch of the kernel in `role` from the committed ncu summary
    ``profiles/<role>_<workload>.md``, if it was taken on the current kernel sources
    (``kernel_source_sha256`` line, over `sources`); else None."""
    p = os.path.join(ROOT, "profiles", f"{role}_{workload_name}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"traffic_bytes_per_full_launch:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash(sources):
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """Samples SM clock, power and clock-event reasons of the benchmarked GPU while the timed region runs.

    Read-only NVML queries through ctypes (libnvidia-ml ships with the driver); falls back to an
    ``nvidia-smi -lms`` subprocess.  Changes no setting."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.01):
        self.samples = []
        self.period = period_s
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        self.source = None
        try:
            import torch

            props = torch.cuda.get_device_properties(device_index)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                raise RuntimeError("handle")
            self._nvml, self._handle = nv, h
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.source = "nvml"
        except Exception:
            self.source = "nvidia-smi"
            self._bus = None

    class _Util(ctypes.Structure):
        _fields_ = [("gpu", ctypes.c_uint), ("memory", ctypes.c_uint)]

    def _sample_nvml(self):
        nv, h = self._nvml, self._handle
        clk, pw, rs, ut = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong(), self._Util()
        while not self._stop.is_set():
            ok = nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0
            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            self._reasons_fn(h, ctypes.byref(rs))
            util = ut.gpu if nv.nvmlDeviceGetUtilizationRates(h, ctypes.byref(ut)) == 0 else -1
            if ok:
                self.samples.append((clk.value, pw.value / 1000.0, int(rs.value), util))
            time.sleep(self.period)

    def start(self):
        if self.source == "nvml":
            self._thread = threading.Thread(target=self._sample_nvml, daemon=True)
            self._thread.start()
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                     "utilization.gpu", "--format=csv,noheader,nounits", "-lms", "50"], stdout=subprocess.PIPE,
                    text=True)
            except Exception:
                self._proc = None

    def stop(self):
        if self.source == "nvml":
            self._stop.set()
            self._thread.join()
        elif getattr(self, "_proc", None) is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            for line in out.splitlines():
                try:
                    c, m, p, r, u = [x.strip() for x in line.split(",")]
                    self.samples.append((float(c), float(p), int(r, 16), float(u)))
                    self.max_mhz = float(m)
                except Exception:
                    pass

    def summary(self):
        """Median SM clock over the samples taken while the GPU was busy (all samples if utilisation is not
        readable), the clock-event reasons seen in any sample, and the sample counts."""
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "samples_under_load": 0, "source": self.source}
        loaded = [s for s in self.samples if s[3] > 0]
        readable = any(s[3] >= 0 for s in self.samples)
        basis = loaded if loaded else self.samples
        bits = 0
        for s in self.samples:
            bits |= s[2]
        reasons = [n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(s[0] for s in basis), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "samples_under_load": len(loaded) if readable else None,
                "sm_mhz_min": min(s[0] for s in basis), "power_w_max": max(s[1] for s in self.samples),
                "period_ms": self.period * 1e3, "source": self.source}


# ---- the CUDA arm -----------------------------------------------------------------------------------------
class Step:
    """Device buffers of one workload and the calls of one step, through the public binding."""

    def __init__(self, w: W.Workload, device, pool_cache=None):
        import torch

        import gated_deltanet_linear_mtp_gb300 as gdn

        self.gdn, self.torch, self.w = gdn, torch, w
        x = w.small_arrays()
        key = (w.state_dtype, w.seed if w.pool_seed is None else w.pool_seed, w.num_slots, w.HV, w.DV, w.DK)
        if pool_cache is not None and key in pool_cache:
            x["pool"] = pool_cache[key]
        else:
            x["pool"] = w.pool()
            if pool_cache is not None:  # sweep points of one state dtype share one pool draw
                pool_cache.clear()
                pool_cache[key] = x["pool"]
        self.x = x
        active = x["indices"] >= 0
        self.A = int(active.sum())
        self.accepted = int(x["accept_len"][active].sum())

        def t(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
            return torch.from_numpy(a).to(device)

        self.d = {k: t(v) for k, v in x.items()}
        # one-pass steps: the tokens of the previous step (its k, v, a, b, accept lengths), committed first
        self.prev, self.prev_accepted = None, 0
        if w.commit_mode == "fused":
            xp = W.previous_step(w)
            self.prev = {k: t(v) for k, v in xp.items()}
            self.prev_accepted = int(xp["accept_len"][active].sum())
        td = {"f32": torch.float32, "bf16": torch.bfloat16}
        self.o = torch.empty((w.B, w.T, w.HV, w.DV), dtype=td[w.out_dtype], device=device)
        self.cache = (torch.empty((w.B, w.T, w.HV, w.DV, w.DK), dtype=td[w.state_dtype], device=device)
                      if w.cache else None)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self._init_e2e(x, device)

    def _init_e2e(self, x, device):
        """End-to-end leg: each step's inputs packed in one pinned host buffer (one copy in), o copied back;
        two device slots of inputs and outputs so that a step's copies overlap its neighbours' compute.
        The steps rotate over disjoint sets of pool slots (same padding positions), so consecutive steps
        touch different states."""
        torch, w = self.torch, self.w
        self.step_keys = ["q", "k", "v", "a", "b", "indices"] + (["accept_len"] if w.commit else [])
        host = {k: self.d[k].cpu() for k in self.step_keys}
        self.layout, off = {}, 0
        for k in self.step_keys:
            nb = host[k].numel() * host[k].element_size()
            self.layout[k] = (off, nb, host[k].dtype, tuple(host[k].shape))
            off = (off + nb + 255) // 256 * 256
        self.packed_bytes = off
        idx = x["indices"]
        act = np.flatnonzero(idx >= 0)
        used = set(idx[act].tolist())
        free = np.random.default_rng([w.seed, 99]).permutation([s for s in range(w.num_slots) if s not in used])
        nsets = 1 + (min(3, len(free) // len(act)) if len(act) else 0)
        self.h_sets = []
        for j in range(nsets):
            buf = torch.empty(self.packed_bytes, dtype=torch.uint8).pin_memory()
            for k in self.step_keys:
                o, nb, dt, shape = self.layout[k]
                src = host[k]
                if k == "indices" and j > 0:
                    src = src.clone()
                    src[torch.from_numpy(act)] = torch.from_numpy(free[(j - 1) * len(act):j * len(act)].astype(np.int32))
                buf[o:o + nb].copy_(src.reshape(-1).view(torch.uint8))
            self.h_sets.append(buf)
        # input / output slots in flight: 2; a one-pass step also reads the previous step's inputs, so 3
        self.nslots = 3 if w.commit_mode == "fused" else 2
        self.dev_slots = [torch.empty(self.packed_bytes, dtype=torch.uint8, device=device)
                          for _ in range(self.nslots)]
        for buf in self.dev_slots:  # every slot holds a valid step (the first one-pass step reads the last slot)
            buf.copy_(self.h_sets[0].to(device))
        self.slot_views = []
        for buf in self.dev_slots:
            v = dict(self.d)
            for k in self.step_keys:
                o, nb, dt, shape = self.layout[k]
                v[k] = buf[o:o + nb].view(dt).view(shape)
            self.slot_views.append(v)
        self.o_slots = [torch.empty_like(self.o) for _ in range(self.nslots)]
        self.h_out = [torch.empty(self.o.shape, dtype=self.o.dtype).pin_memory() for _ in range(self.nslots)]
        self.h2d_bytes = sum(self.layout[k][1] for k in self.step_keys)
        self.d2h_bytes = self.o.numel() * self.o.element_size()
        self.e2e_sets = nsets

    def recurrent(self, d=None, o=None, prev=None):
        d, w, o = d or self.d, self.w, self.o if o is None else o
        if w.commit_mode == "fused":
            pv = prev or self.prev
            self.gdn.gdn_mtp_verify_commit(
                self.gdn.ReplayTokens(pv["k"], pv["v"], pv["a"], pv["b"], pv["accept_len"]), d["q"], d["k"], d["v"],
                d["a"], d["b"], d["A_log"], d["dt_bias"], d["pool"], d["indices"], o, self.err, scale=w.scale,
                l2_eps=w.l2_eps)
        elif w.mode == "decode":
            self.gdn.gdn_decode(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["pool"],
                                d["indices"], o, self.err, scale=w.scale, l2_eps=w.l2_eps)
        else:
            self.gdn.gdn_mtp_verify(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["pool"],
                                    d["indices"], o, self.cache, self.err, scale=w.scale, l2_eps=w.l2_eps)

    def commit(self, d=None):
        if not self.w.commit or self.w.commit_mode == "fused":  # a one-pass step commits inside recurrent()
            return
        d, w = d or self.d, self.w
        if w.commit_mode == "replay":
            self.gdn.gdn_commit_replay(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["pool"],
                                       d["indices"], d["accept_len"], self.err, scale=w.scale, l2_eps=w.l2_eps)
        else:
            self.gdn.gdn_commit(d["pool"], d["indices"], self.cache, d["accept_len"], self.err)

    E2E_GRAPH_STEPS = 32

    def run_e2e(self, K: int, warmup: int, comp, min_seconds: float = 0.0):
        """Pipelined steps through the public calls, captured once as a CUDA graph of E2E_GRAPH_STEPS steps and
        replayed at least K steps and at least `min_seconds`; returns (device time per step in ms, from before
        the first copy in to after the last copy out; steps timed).  Step i: copy in (H2D stream) ->
        verify/decode + commit (compute stream) -> copy o out (D2H stream); step i+1's copy in runs during
        step i's compute."""
        torch = self.torch
        G = self.E2E_GRAPH_STEPS
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        NSL = self.nslots
        fused = self.w.commit_mode == "fused"
        up = [torch.cuda.Event() for _ in range(NSL)]
        done = [torch.cuda.Event() for _ in range(NSL)]
        down = [torch.cuda.Event() for _ in range(NSL)]

        def steps(cs):
            h2d.wait_stream(cs)
            d2h.wait_stream(cs)
            for i in range(G):
                s = i % NSL
                last_reader = i - NSL + (1 if fused else 0)  # the last step reading this input slot
                if last_reader >= 0:
                    h2d.wait_event(done[last_reader % NSL])
                with torch.cuda.stream(h2d):
                    self.dev_slots[s].copy_(self.h_sets[i % len(self.h_sets)], non_blocking=True)
                    up[s].record(h2d)
                cs.wait_event(up[s])
                if i >= NSL:
                    cs.wait_event(down[s])  # the o of step i - NSL has been copied out of this output slot
                with torch.cuda.stream(cs):
                    self.recurrent(self.slot_views[s], self.o_slots[s], self.slot_views[(i - 1) % NSL])
                    self.commit(self.slot_views[s])
                    done[s].record(cs)
                d2h.wait_event(done[s])
                with torch.cuda.stream(d2h):
                    self.h_out[s].copy_(self.o_slots[s], non_blocking=True)
                    down[s].record(d2h)
            cs.wait_stream(h2d)
            cs.wait_stream(d2h)

        for _ in range(max(1, warmup // G)):  # eager warm-up
            steps(comp)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(comp)
        with torch.cuda.graph(graph, stream=cap):
            steps(cap)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(comp):
            t0.record(comp)
            graph.replay()
            t1.record(comp)
        torch.cuda.synchronize()
        one_ms = max(t0.elapsed_time(t1), 1e-3)
        reps = max(1, -(-K // G), int(math.ceil(min_seconds * 1e3 / one_ms)))
        with torch.cuda.stream(comp):
            t0.record(comp)
            for _ in range(reps):
                graph.replay()
            t1.record(comp)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / (reps * G), reps * G

    @property
    def launches_per_step(self) -> int:
        return 1 + (1 if self.w.commit and self.w.commit_mode != "fused" else 0)


_POOL_CACHE: dict = {}
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e nominal (~8 TB/s); the specification's >= 70 % target is against it
MIN_WINDOW_S = 1.0        # each point's timed region covers at least this much device time


def roofline_block(kernel: dict, peak: float, peak_src: str, traffic) -> dict:
    """Roofline of the dominant kernel: against the measured copy peak (frac) and the nominal 8 TB/s
    (frac_nominal, the basis of the >= 0.70 target)."""
    return {
        "kernel": f"{kernel['kernel']} ({kernel['role']})",
        "bound": "hbm",
        "achieved": kernel["achieved_gbs"],
        "peak": peak,
        "unit": "GB/s",
        "frac": kernel["frac"],
        "peak_source": peak_src + ", of measured" if peak_src.startswith("measured") else peak_src,
        "nominal_peak": NOMINAL_HBM_GBS,
        "frac_nominal": kernel["achieved_gbs"] / NOMINAL_HBM_GBS,
        "target_basis": "frac_nominal (>= 0.70 of the nominal ~8 TB/s on verify T=4 B=128 bf16 state)",
        "algorithmic_bytes_per_launch": kernel["algorithmic_bytes"],
        "avg_launch_us": kernel["avg_us"],
        "traffic": traffic,
    }


class _Flush:
    """Write a buffer larger than L2 (evicts everything), then read another one so that the lines left in L2
    are clean and the timed step does not pay for writing the flush's dirty lines back."""

    def __init__(self, device):
        import torch

        props = torch.cuda.get_device_properties(device)
        n = max(256 << 20, 2 * props.L2_cache_size) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.zeros(n, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.fill_(1.0)
        self.r.sum()


def measure_point(args, w: W.Workload, rank: int, world: int, local_rank: int, dist, min_seconds: float,
                  e2e: bool = True, steps: int = None) -> dict:
    """One workload on this rank's GPU: W warm-up steps, then R x K timed steps (R chosen from the warm-up
    so that the timed region covers at least `min_seconds` of device time; the same R on every rank), each
    step bracketed by CUDA events with an L2 flush before it, outside the events.  Then the end-to-end leg
    (`e2e`).  Returns the result record (no CPU baseline)."""
    import torch

    device = torch.device("cuda", local_rank)
    K = args.steps if steps is None else steps
    wr = rank_workload(w, rank)
    st = Step(wr, device, _POOL_CACHE if w.pool_seed is not None else None)
    flush = _Flush(device)
    stream = torch.cuda.current_stream(device)

    def one(ev=None):
        flush()
        if ev is not None:
            ev[0].record(stream)
        st.recurrent()
        if ev is not None:
            ev[1].record(stream)
        st.commit()
        if ev is not None:
            ev[2].record(stream)

    wev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.warmup)]
    for i in range(args.warmup):
        one(wev[i])
    torch.cuda.synchronize()
    if st.err.item() != 0:
        raise RuntimeError(f"device error word {st.err.item()} after warm-up ({w.name})")
    warm_ms = statistics.median(e[0].elapsed_time(e[2]) for e in wev)
    R = max(1, int(math.ceil(min_seconds * 1e3 / max(K * warm_ms, 1e-6))))
    R = int(max_over_ranks(R, dist, device))
    n = R * K
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    sampler = ClockSampler(local_rank)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_wall = time.perf_counter()
    for i in range(n):
        one(evs[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    sampler.stop()
    if dist is not None:
        dist.barrier()
    if st.err.item() != 0:
        raise RuntimeError(f"device error word {st.err.item()} after the timed steps ({w.name})")
    rec_ms = [e[0].elapsed_time(e[1]) for e in evs]
    com_ms = [e[1].elapsed_time(e[2]) for e in evs]
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms), dist, device)
    tokens_all = sum_over_ranks(st.A * wr.T * n, dist, device)

    e2e_rec = None
    if e2e:
        if dist is not None:
            dist.barrier()
        e2e_ms, e2e_steps = st.run_e2e(K, args.warmup, stream, min_seconds)
        e2e_ms_step = max_over_ranks(e2e_ms, dist, device)
        if st.err.item() != 0:
            raise RuntimeError(f"device error word {st.err.item()} after the end-to-end leg ({w.name})")
        e2e_rec = {"value": sum_over_ranks(st.A * wr.T, dist, device) / (e2e_ms_step * 1e-3), "unit": "tokens/s",
                   "h2d_bytes_per_step": st.h2d_bytes, "d2h_bytes_per_step": st.d2h_bytes,
                   "ms_per_step": e2e_ms_step, "timed_steps": e2e_steps}

    peak, peak_src = hbm_peak()
    fused = wr.commit_mode == "fused"
    rb = fused_bytes(wr, st.A, st.prev_accepted) if fused else recurrent_bytes(wr, st.A)
    cb = commit_bytes(wr, st.A, st.accepted) if wr.commit and not fused else 0
    role = "decode" if w.mode == "decode" else ("verify_commit" if fused else "verify")
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    kernels = [{"role": role, "kernel": kernel_name(wr, role, sms), "avg_us": statistics.mean(rec_ms) * 1e3,
                "algorithmic_bytes": rb}]
    if wr.commit and not fused:
        crole = "commit_replay" if wr.commit_mode == "replay" else "commit"
        kernels.append({"role": crole, "kernel": kernel_name(wr, crole, sms),
                        "avg_us": statistics.mean(com_ms) * 1e3, "algorithmic_bytes": cb})
    for k in kernels:
        k["achieved_gbs"] = k["algorithmic_bytes"] / (k["avg_us"] * 1e-6) / 1e9
        k["frac"] = k["achieved_gbs"] / peak
        k["frac_nominal"] = k["achieved_gbs"] / NOMINAL_HBM_GBS
    dom = max(kernels, key=lambda k: k["avg_us"])
    props = torch.cuda.get_device_properties(device)
    result = {
        "metric": METRIC,
        "value": tokens_all / (total_ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "repeats": R,
        "timed_steps": n,
        "warmup": args.warmup,
        "ms_per_step": total_ms / n,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded numpy draws; shapes and distributions of the named workload)",
        "config": {
            "workload": w.name, "B": w.B, "active_lanes": st.A, "T": w.T, "HK": w.HK, "HV": w.HV, "DK": w.DK,
            "DV": w.DV, "num_slots": w.num_slots, "state_dtype": w.state_dtype, "qkv_dtype": w.qkv_dtype,
            "out_dtype": w.out_dtype, "intermediate_cache": w.cache, "commit_per_step": w.commit,
            "step": ("gdn_decode" if w.mode == "decode" else
                     "gdn_mtp_verify_commit (the previous step's accepted prefix committed, then verify)" if fused else
                     "gdn_mtp_verify" + ((" + gdn_commit_replay" if w.commit_mode == "replay" else " + gdn_commit")
                                         if w.commit else "")),
            "l2": "flushed before every step outside its CUDA events (256 MiB write, then 256 MiB read: clean lines)",
            "parallelism": f"replicas x{world} (independent batches, no collective)",
            "timing": (f"CUDA events per step on the launch stream, summed over {R} x {K} steps (the timed region "
                       f"covers >= {min_seconds:g} s of device time); max over ranks"),
            "e2e": (f"pipelined: each step's inputs copied in from pinned host memory (one packed copy) and its o "
                    f"copied back, on H2D / D2H streams beside the compute stream, {st.E2E_GRAPH_STEPS} steps captured "
                    f"as one CUDA graph and replayed for >= {min_seconds:g} s; no L2 flush: steps rotate over "
                    f"{st.e2e_sets} disjoint sets of pool slots") if e2e else None,
        },
        "verify_steps_per_s": n * world / (total_ms * 1e-3),
        "hbm_gbs_step": (rb + cb) * world * n / (total_ms * 1e-3) / 1e9,
        "roofline": roofline_block(dom, peak, peak_src, recorded_traffic(dom["role"], w.name)),
        "kernels": kernels,
        "e2e": e2e_rec,
        "gpu_launches": st.launches_per_step * n,
        "clocks": sampler.summary(),
        "device": props.name,
        "sm_count": props.multi_processor_count,
        "wall_s_timed_region": t_wall,
    }
    del st, flush
    torch.cuda.empty_cache()
    return result


POINT_KEYS = ("value", "unit", "ms_per_step", "repeats", "timed_steps", "verify_steps_per_s", "hbm_gbs_step",
              "roofline", "kernels", "e2e", "gpu_launches", "clocks", "wall_s_timed_region")
# the metric's T = 1 and T = 8 points and the verify + replay-commit and one-pass steps, each measured like the
# main line
POINTS = ("decode", "verify8", "verify4_replay", "verify8_replay", "verify4_fused", "verify8_fused")


def point_record(r: dict) -> dict:
    rec = {k: r[k] for k in POINT_KEYS}
    rec["config"] = {k: r["config"][k] for k in ("workload", "B", "active_lanes", "T", "state_dtype",
                                                   "intermediate_cache", "step")}
    return rec


def sweep_summary(args, rank, world, local_rank, dist, pts, steps: int) -> list:
    """Tokens/s and the dominant kernel's fraction of the measured peak per point (fixed step count, no
    end-to-end leg)."""
    out = []
    for w in pts:
        r = measure_point(args, w, rank, world, local_rank, dist, 0.0, e2e=False, steps=steps)
        out.append({"workload": w.name, "B": w.B, "T": w.T, "state_dtype": w.state_dtype,
                    "tokens_per_s": r["value"], "ms_per_step": r["ms_per_step"],
                    "kernel": r["roofline"]["kernel"], "frac": r["roofline"]["frac"],
                    "frac_nominal": r["roofline"]["frac_nominal"], "sm_mhz": r["clocks"]["sm_mhz"]})
    return out


def run_cuda_arm(args, w: W.Workload, rank: int, world: int, local_rank: int, emit=True, points=(),
                 sweep_steps: int = 0):
    import torch

    torch.cuda.set_device(local_rank)
    dist = init_dist(world, "nccl")
    result = measure_point(args, w, rank, world, local_rank, dist, args.min_seconds)
    if points:
        result["points"] = {}
        for name in points:
            pw = W.NAMED[name]()
            result["points"][pw.name] = point_record(
                measure_point(args, pw, rank, world, local_rank, dist, args.min_seconds))
    if sweep_steps > 0:
        result["sweep"] = {"steps_per_point": sweep_steps,
                           "points": sweep_summary(args, rank, world, local_rank, dist, W.sweep(), sweep_steps)}
    if rank == 0 and not args.no_cpu_baseline and emit:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0 and emit:
        print(json.dumps(result), flush=True)
    return result


# ---- prefill and the gated RMSNorm ----------------------------------------------------------------------
PREFILL_METRIC = "GDN prefill tokens/s (variable-length prompts into the state pool)"
NORM_METRIC = "GDN gated RMSNorm rows/s and achieved HBM GB/s"
FP32_LANES_PER_SM = 128  # FP32 FMA lanes per Blackwell SM
PREFILL_FLOPS_PER_ELEM = 7  # per state element and token: decay 1, S.kh 2, rank-1 update 2, S.qh 2


PREFILL_CHUNK = 32  # tokens per chunk of the chunked prefill


def prefill_is_chunked(pw) -> bool:
    return pw.DK in (64, 128)


def prefill_mma_flops(pw, x):
    """tcgen05 MMA flops the chunked prefill issues per launch on its TMA path (bf16 q, k, v, DV >= 128), counted
    from the MMA shapes: per item (sequence, value head, block of 128 state rows) and chunk of 32 tokens,
    P = S_0 hi and lo against [k; q] (2 x 2*128*64*DK), the Gram product [k; q][k; q]^T (2*128*64*DK, M = 128),
    O = delta KQw^T in three part products (3 x 2*128*32*32), the update in two (2 x 2*128*DK*32).  None
    elsewhere (the token loop, or the chunked kernel's other token path)."""
    if not prefill_is_chunked(pw) or pw.qkv_dtype != "bf16" or pw.DV < 128:
        return None
    per = 2 * 2 * 128 * 64 * pw.DK + 2 * 128 * 64 * pw.DK + 3 * 2 * 128 * 32 * 32 + 2 * 2 * 128 * pw.DK * 32
    lens = np.diff(x["cu_seqlens"])[x["indices"] >= 0]
    chunks = int(((lens + PREFILL_CHUNK - 1) // PREFILL_CHUNK).sum())
    return float(per) * chunks * pw.HV * ((pw.DV + 127) // 128)


def prefill_bytes(pw, x) -> float:
    """What the prefill must move: q, k, v, a, b in and o out for every active token, the state read (sequences with
    an initial state) and written (every active sequence)."""
    isz = 2 if pw.qkv_dtype == "bf16" else 4
    osz = 2 if pw.out_dtype == "bf16" else 4
    ssz = 2 if pw.state_dtype == "bf16" else 4
    act = x["indices"] >= 0
    lens = np.diff(x["cu_seqlens"])
    tokens = int(lens[act].sum())
    nseq = int((act & (lens > 0)).sum())
    nread = int((act & (lens > 0) & (x["has_initial_state"] != 0)).sum())
    per_tok = (2 * pw.HK * pw.DK + pw.HV * pw.DV + 2 * pw.HV) * isz + pw.HV * pw.DV * osz
    state = pw.HV * pw.DV * pw.DK * ssz
    return float(tokens * per_tok + (nseq + nread) * state)


def alu_peak_tflops(sms: int, mhz: float) -> float:
    """FP32 FMA peak of the CUDA cores (not the tensor cores): SMs x 128 lanes x 2 flops x clock."""
    return sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def _timed_calls(call, K: int, warmup: int, stream, sampler, min_seconds: float = 0.0):
    """W warm-up calls, then R x K timed calls (R from the warm-up, so that the timed calls cover at least
    `min_seconds` of device time), each bracketed by CUDA events; returns (per-call ms, wall seconds)."""
    import torch

    wev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(warmup)]
    for i in range(warmup):
        wev[i][0].record(stream)
        call()
        wev[i][1].record(stream)
    torch.cuda.synchronize()
    warm_ms = statistics.median(e[0].elapsed_time(e[1]) for e in wev) if wev else 0.0
    K = K * max(1, int(math.ceil(min_seconds * 1e3 / max(K * warm_ms, 1e-6)))) if min_seconds > 0 else K
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler.start()
    t_wall = time.perf_counter()
    for i in range(K):
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    sampler.stop()
    return [e[0].elapsed_time(e[1]) for e in evs], t_wall


def _prefill_pairs(pw, x):
    """(prompt, value head) pairs of the active prompts, in order."""
    return [(b, h) for b in range(pw.B) if x["indices"][b] >= 0 for h in range(pw.HV)]


def _prefill_pair(orc, pw, x, b: int, h: int, max_tokens=None):
    """The oracle's prefill of prompt b, value head h alone (its first max_tokens tokens if given), on a copy
    of its slot; returns the tokens run."""
    cu = x["cu_seqlens"]
    lo, hi, hk, slot = int(cu[b]), int(cu[b + 1]), h // (pw.HV // pw.HK), int(x["indices"][b])
    if max_tokens is not None:
        hi = min(hi, lo + max_tokens)
    d = dict(T=0, HK=1, HV=1, DK=pw.DK, DV=pw.DV, num_slots=1, qkv_dtype=pw.qkv_dtype, state_dtype=pw.state_dtype,
             scale=pw.scale, l2_eps=pw.l2_eps)
    y = dict(q=np.ascontiguousarray(x["q"][lo:hi, hk:hk + 1]), k=np.ascontiguousarray(x["k"][lo:hi, hk:hk + 1]),
             v=np.ascontiguousarray(x["v"][lo:hi, h:h + 1]), a=np.ascontiguousarray(x["a"][lo:hi, h:h + 1]),
             b=np.ascontiguousarray(x["b"][lo:hi, h:h + 1]), A_log=np.ascontiguousarray(x["A_log"][h:h + 1]),
             dt_bias=np.ascontiguousarray(x["dt_bias"][h:h + 1]), indices=np.zeros(1, np.int32))
    pool = np.ascontiguousarray(x["pool"][slot:slot + 1, h:h + 1])
    orc.prefill(d, y, np.array([0, hi - lo], np.int32), pool, np.array([x["has_initial_state"][b]], np.int32))
    return hi - lo


def _prefill_cpu_baseline(pw, x, seconds: float):
    """The oracle as it stands (fp64 C loops) on (prompt, head) pairs in order -- each a whole prompt for one
    value head -- on every host core until about `seconds` have passed (and on one thread beside it);
    tokens/s of the layer = pair tokens / HV / time (a token's work is HV such pairs)."""
    import oracle

    orc = oracle.default()
    pairs = _prefill_pairs(pw, x)
    cores = host_cores()
    cu = x["cu_seqlens"]
    ntok = [int(cu[b + 1] - cu[b]) for b, _ in pairs]
    work = [(lambda b=b, h=h: _prefill_pair(orc, pw, x, b, h)) for b, h in pairs]
    n1, dt1 = oracle_throughput(work, seconds / 3.0, 1)
    n, dt = oracle_throughput(work, seconds * 2.0 / 3.0, cores)
    tok1, tok = sum(ntok[:n1]), sum(ntok[:n])
    return {"value": tok / pw.HV / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "one_thread": {"value": tok1 / pw.HV / dt1, "unit": "tokens/s", "pairs": n1, "seconds": dt1},
            "sample": f"oracle prefill of the first {n} of {len(pairs)} (prompt, value head) pairs of {pw.name} "
                      f"({tok} pair-tokens), fp64 C loops on {cores} threads, {dt:.1f} s; tokens/s = pair-tokens / "
                      f"HV / time; one thread: {n1} pairs in {dt1:.1f} s"}


def run_prefill_arm(args, pw, rank: int, world: int, local_rank: int):
    import torch

    import gated_deltanet_linear_mtp_gb300 as gdn

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = init_dist(world, "nccl")
    pr = pw if rank == 0 else pw.replace(seed=pw.seed + 7919 * rank)
    x = pr.arrays()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    t = {k: to_dev(v) for k, v in x.items()}
    N = int(x["cu_seqlens"][-1])
    odt = torch.bfloat16 if pw.out_dtype == "bf16" else torch.float32
    o = torch.empty((N, pw.HV, pw.DV), dtype=odt, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    names = ("q", "k", "v", "a", "b")

    def call(src=t, out=o):
        gdn.gdn_prefill(src["q"], src["k"], src["v"], src["a"], src["b"], t["A_log"], t["dt_bias"], t["pool"],
                        t["indices"], t["cu_seqlens"], out, t["has_initial_state"], err, scale=pw.scale,
                        l2_eps=pw.l2_eps)

    sampler = ClockSampler(local_rank)
    if dist is not None:
        dist.barrier()
    ms, t_wall = _timed_calls(call, args.steps, args.warmup, stream, sampler, args.min_seconds)
    if err.item() != 0:
        raise RuntimeError(f"device error word {err.item()}")
    total_ms = max_over_ranks(sum(ms), dist, device)
    n_timed = len(ms)
    lens = np.diff(x["cu_seqlens"])
    active_tokens = int(lens[x["indices"] >= 0].sum())
    tokens_all = sum_over_ranks(active_tokens * n_timed, dist, device)

    # end to end through the binding: each step's q, k, v, a, b copied in from pinned host memory and o
    # copied back, on the compute stream
    host_in = {k: t[k].cpu().pin_memory() for k in names}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = o.numel() * o.element_size()

    def e2e_step():
        for k in names:
            t[k].copy_(host_in[k], non_blocking=True)
        call()
        o_host.copy_(o, non_blocking=True)

    K_e2e = max(3, min(args.steps, 20))
    e2e_ms, _ = _timed_calls(e2e_step, K_e2e, 2, stream, ClockSampler(local_rank))
    e2e_ms_step = max_over_ranks(statistics.mean(e2e_ms), dist, device)

    props = torch.cuda.get_device_properties(device)
    clocks = sampler.summary()
    max_mhz = clocks.get("sm_max_mhz") or 2070.0
    avg_us = statistics.mean(ms) * 1e3
    flops = PREFILL_FLOPS_PER_ELEM * pw.DV * pw.DK * pw.HV * active_tokens
    achieved = flops / (avg_us * 1e-6) / 1e12
    if prefill_is_chunked(pw):
        # the chunked kernel: contractions on the tensor cores; the method's flops against the bf16 tensor peak,
        # with the MMA flops it issues and the HBM fraction of what it must move beside them
        peak, peak_src = tensor_peak()
        mma = prefill_mma_flops(pw, x)
        pb = prefill_bytes(pw, x)
        hbm, hbm_src = hbm_peak()
        roof = {"kernel": "gdn_prefill_chunked_kernel", "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_src,
                "algorithmic_flops_per_launch": flops, "avg_launch_us": avg_us,
                "mma_flops_per_launch": mma,
                "mma_tflops": None if mma is None else mma / (avg_us * 1e-6) / 1e12,
                "mma_frac": None if mma is None else mma / (avg_us * 1e-6) / 1e12 / peak,
                "hbm": {"algorithmic_bytes_per_launch": pb, "achieved_gbs": pb / (avg_us * 1e-6) / 1e9,
                        "peak_gbs": hbm, "frac": pb / (avg_us * 1e-6) / 1e9 / hbm, "peak_source": hbm_src},
                "limited_by": "the chain of chunks of each (sequence, head): one CTA per SM works through its item's "
                              "32-token chunks in order, so the per-chunk latency, not a unit's throughput, sets the "
                              "time",
                "traffic": recorded_traffic("prefill", pw.name, PREFILL_SOURCES)}
    else:
        peak = alu_peak_tflops(props.multi_processor_count, max_mhz)
        roof = {"kernel": "gdn_prefill_kernel", "bound": "alu", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"derived: {props.multi_processor_count} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 "
                               f"flops x {max_mhz:.0f} MHz (maximum SM clock)",
                "algorithmic_flops_per_launch": flops, "avg_launch_us": avg_us,
                "traffic": recorded_traffic("prefill", pw.name, PREFILL_SOURCES)}
    result = {
        "metric": PREFILL_METRIC, "value": tokens_all / (total_ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "timed_steps": n_timed, "warmup": args.warmup, "ms_per_step": total_ms / n_timed,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy draws; shapes and distributions of the named workload)",
        "config": {"workload": pw.name, "B": pw.B, "tokens": N, "active_tokens": active_tokens, "HK": pw.HK,
                   "HV": pw.HV, "DK": pw.DK, "DV": pw.DV, "state_dtype": pw.state_dtype, "qkv_dtype": pw.qkv_dtype,
                   "fresh_sequences": int((x["has_initial_state"] == 0).sum()),
                   "step": "gdn_prefill (every prompt from its slot or from zero; final state into the slot)",
                   "l2": f"not flushed: the step reads {h2d / 1e9:.2f} GB of token inputs, more than L2",
                   "parallelism": f"replicas x{world} (independent prompts, no collective)",
                   "timing": f"CUDA events per call on the launch stream, summed over {n_timed} calls (>= "
                             f"{args.min_seconds:g} s of device time); max over ranks",
                   "e2e": "inputs copied in from pinned host memory and o copied back on the compute stream, "
                          "per step, not overlapped"},
        "roofline": roof,
        "e2e": {"value": sum_over_ranks(active_tokens, dist, device) / (e2e_ms_step * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_step},
        "gpu_launches": n_timed, "clocks": clocks, "device": props.name,
        "sm_count": props.multi_processor_count, "wall_s_timed_region": t_wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = _prefill_cpu_baseline(pw, x, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    return result


def run_norm_arm(args, rank: int, world: int, local_rank: int, rows: int = 65536 * 32, DV: int = 128):
    """The gated RMSNorm over the outputs of the ISL-8K prefill (65,536 tokens x 32 heads of 128, bf16)."""
    import torch

    import gated_deltanet_linear_mtp_gb300 as gdn

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = init_dist(world, "nccl")
    g = W.gated_norm_inputs(rows, DV, "bf16", "bf16", seed=17 + 7919 * rank)
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)  # noqa: E731
    o, z = bf(g["o"]), bf(g["z"])
    wt = torch.from_numpy(g["w"]).to(device)
    y = torch.empty_like(o)
    stream = torch.cuda.current_stream(device)
    sampler = ClockSampler(local_rank)
    if dist is not None:
        dist.barrier()
    ms, t_wall = _timed_calls(lambda: gdn.gdn_gated_rmsnorm(o, z, wt, y), args.steps, args.warmup, stream, sampler,
                              args.min_seconds)
    total_ms = max_over_ranks(sum(ms), dist, device)
    n_timed = len(ms)
    nbytes = rows * DV * 2 * 3 + DV * 4
    avg_us = statistics.mean(ms) * 1e3
    peak, peak_src = hbm_peak()
    achieved = nbytes / (avg_us * 1e-6) / 1e9
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    z_host = torch.empty(z.shape, dtype=z.dtype).pin_memory()
    o_host.copy_(o)
    z_host.copy_(z)
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()

    def e2e_step():
        o.copy_(o_host, non_blocking=True)
        z.copy_(z_host, non_blocking=True)
        gdn.gdn_gated_rmsnorm(o, z, wt, y)
        y_host.copy_(y, non_blocking=True)

    e2e_ms, _ = _timed_calls(e2e_step, max(3, min(args.steps, 20)), 2, stream, ClockSampler(local_rank))
    e2e_ms_step = max_over_ranks(statistics.mean(e2e_ms), dist, device)
    props = torch.cuda.get_device_properties(device)
    result = {
        "metric": NORM_METRIC, "value": rows * n_timed * world / (total_ms * 1e-3), "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "timed_steps": n_timed, "warmup": args.warmup,
        "ms_per_step": total_ms / n_timed,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy draws)",
        "config": {"workload": f"gated_rmsnorm_rows{rows}_DV{DV}_bf16", "rows": rows, "DV": DV,
                   "o_dtype": "bf16", "z_dtype": "bf16",
                   "l2": f"not flushed: each call moves {nbytes / 1e9:.2f} GB, more than L2",
                   "parallelism": f"replicas x{world}", "timing": "CUDA events per call, summed; max over ranks",
                   "e2e": "o and z copied in from pinned host memory and y copied back per step"},
        "roofline": {"kernel": "gdn_gated_rmsnorm_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src + ", of measured" if peak_src.startswith("measured") else peak_src,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": nbytes, "avg_launch_us": avg_us,
                     "traffic": recorded_traffic("gated_norm", f"gated_rmsnorm_rows{rows}_DV{DV}_bf16", NORM_SOURCES)},
        "e2e": {"value": rows * world / (e2e_ms_step * 1e-3), "unit": "rows/s",
                "h2d_bytes_per_step": 2 * rows * DV * 2, "d2h_bytes_per_step": rows * DV * 2,
                "ms_per_step": e2e_ms_step},
        "gpu_launches": n_timed, "clocks": sampler.summary(), "device": props.name,
        "sm_count": props.multi_processor_count, "wall_s_timed_region": t_wall,
    }
    if rank == 0:
        print(json.dumps(result), flush=True)
    return result


IN_PROJ_METRIC = "GDN in_proj + causal conv1d rows/s and achieved HBM GB/s"
IN_PROJ_NAMED = {"in_proj16": W.in_proj_verify16, "in_proj8": W.in_proj_decode8, "in_proj512": W.in_proj_verify512}
IN_PROJ_DECODE = {"in_proj8"}  # decode rows (the state is written back); the others are verify rows (records)
IN_PROJ_SOURCES = ["gated_deltanet_linear_mtp_gb300/csrc/gdn_in_proj_conv.cu",
                   "gated_deltanet_linear_mtp_gb300/csrc/gdn_tcgen05.cuh",
                   "gated_deltanet_linear_mtp_gb300/csrc/gdn_common.cuh"]


def in_proj_counts(w: W.InProjWorkload, active: int, decode: bool):
    """(algorithmic bytes, flops) of one call: W once, the active lanes' x rows, outputs, state read (and
    written back, or the records), the taps; flops = 2 x rows x C x H of the projection (the convolution's
    2 K per convolved output is counted too)."""
    ob = 2 if w.out_dtype == "bf16" else 4
    sb = 2 if w.conv_dtype == "bf16" else 4
    rows = active * w.T
    nbytes = (w.C * w.H * 2 + rows * w.H * 2 + rows * w.C * ob + active * (w.K - 1) * w.Cc * sb
              + (active * (w.K - 1) * w.Cc * sb if decode else rows * w.Cc * sb) + w.Cc * (w.K + 1) * 4
              + w.B * 4)
    flops = 2 * rows * w.C * w.H + 2 * w.K * rows * w.Cc
    return nbytes, flops


def run_in_proj_arm(args, name: str, rank: int, world: int, local_rank: int):
    """The in_proj projection with its conv1d epilogue on one workload: L2 flushed before every timed call (W, 50
    MB, would otherwise stay in L2), CUDA events around the call alone."""
    import torch

    import gated_deltanet_linear_mtp_gb300 as gdn

    w = IN_PROJ_NAMED[name]().replace(seed=IN_PROJ_NAMED[name]().seed + 7919 * rank)
    decode = name in IN_PROJ_DECODE
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = init_dist(world, "nccl")
    x = w.arrays()

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    d = {k: t(v) for k, v in x.items()}
    odt = torch.bfloat16 if w.out_dtype == "bf16" else torch.float32
    B, T = w.B, w.T
    out = gdn.InProjOut(*(torch.empty(s, dtype=odt, device=device) for s in
                          ((B, T, w.HK, w.DK), (B, T, w.HK, w.DK), (B, T, w.HV, w.DV), (B, T, w.HV, w.DV),
                           (B, T, w.HV), (B, T, w.HV))))
    rec = None if decode else torch.empty((B, T, w.Cc), dtype=d["conv_state"].dtype, device=device)

    def call():
        gdn.gdn_in_proj_conv(d["x"], d["W"], d["conv_w"], d["conv_b"], d["conv_state"], d["indices"], out, decode,
                             rec, silu=w.silu)

    stream = torch.cuda.current_stream(device)
    flush = _Flush(device)
    sampler = ClockSampler(local_rank)
    for _ in range(args.warmup):
        flush()
        call()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    n_timed = max(args.steps, 1)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_timed)]
    sampler.start()
    t_wall = time.perf_counter()
    for e in evs:
        flush()
        e[0].record(stream)
        call()
        e[1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    sampler.stop()
    ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = max_over_ranks(sum(ms), dist, device)
    active = int((x["indices"] >= 0).sum())
    nbytes, flops = in_proj_counts(w, active, decode)
    avg_us = statistics.mean(ms) * 1e3
    peak, peak_src = hbm_peak()
    tpeak, tpeak_src = tensor_peak()
    achieved = nbytes / (avg_us * 1e-6) / 1e9
    tflops = flops / (avg_us * 1e-6) / 1e12
    hbm_frac, tensor_frac = achieved / peak, tflops / tpeak
    bound = "hbm" if hbm_frac >= tensor_frac else "tensor"
    # end to end: x in from pinned host memory, the six outputs (and the records) back, every step
    x_host = torch.empty(d["x"].shape, dtype=d["x"].dtype).pin_memory()
    x_host.copy_(d["x"])
    outs = [out.q, out.k, out.v, out.z, out.b, out.a] + ([] if rec is None else [rec])
    back = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]

    def e2e_step():
        d["x"].copy_(x_host, non_blocking=True)
        call()
        for h, o in zip(back, outs):
            h.copy_(o, non_blocking=True)

    e2e_ms, _ = _timed_calls(e2e_step, max(3, min(args.steps, 50)), 3, stream, ClockSampler(local_rank))
    e2e_ms_step = max_over_ranks(statistics.mean(e2e_ms), dist, device)
    h2d = x_host.numel() * 2
    d2h = sum(o.numel() * o.element_size() for o in outs)
    props = torch.cuda.get_device_properties(device)
    rows = active * T
    result = {
        "metric": IN_PROJ_METRIC, "value": rows * n_timed * world / (total_ms * 1e-3), "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "timed_steps": n_timed, "warmup": args.warmup,
        "ms_per_step": total_ms / n_timed, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 x bf16 -> f32", "data": "synthetic (seeded numpy draws, random-init weights)",
        "config": {"workload": w.name, "B": B, "T": T, "rows": rows, "H": w.H, "C": w.C, "Cc": w.Cc, "K": w.K,
                   "HK": w.HK, "HV": w.HV, "DK": w.DK, "DV": w.DV, "conv_dtype": w.conv_dtype,
                   "out_dtype": w.out_dtype, "mode": "decode (state written back)" if decode else
                   "verify (state read, records written)",
                   "l2": "flushed before every timed call (256 MiB write + read, outside the events)",
                   "parallelism": f"replicas x{world}", "timing": "CUDA events per call, summed; max over ranks",
                   "e2e": "x copied in from pinned host memory and every output copied back per step"},
        "roofline": {"kernel": "gdn_in_proj_conv_kernel", "bound": bound,
                     "achieved": achieved if bound == "hbm" else tflops, "peak": peak if bound == "hbm" else tpeak,
                     "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                     "frac": hbm_frac if bound == "hbm" else tensor_frac,
                     "peak_source": (peak_src if bound == "hbm" else tpeak_src) + ", of measured",
                     "hbm": {"achieved_gbs": achieved, "frac": hbm_frac, "frac_nominal": achieved / NOMINAL_HBM_GBS},
                     "tensor": {"achieved_tflops": tflops, "frac": tensor_frac},
                     "algorithmic_bytes_per_launch": nbytes, "flops_per_launch": flops, "avg_launch_us": avg_us,
                     "traffic": recorded_traffic("in_proj_conv", w.name, IN_PROJ_SOURCES)},
        "e2e": {"value": rows * world / (e2e_ms_step * 1e-3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_step},
        "gpu_launches": n_timed, "clocks": sampler.summary(), "device": props.name,
        "sm_count": props.multi_processor_count, "wall_s_timed_region": t_wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = _in_proj_cpu_baseline(w, x, decode, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    return result


def _in_proj_lane(orc, w, x, b: int, decode: bool):
    """The oracle's in_proj + convolution of lane b alone (on a copy of the state)."""
    d = dict(T=w.T, H=w.H, HK=w.HK, HV=w.HV, DK=w.DK, DV=w.DV, K=w.K, num_slots=w.num_slots, x_dtype="bf16",
             conv_dtype=w.conv_dtype, silu=int(w.silu))
    orc.in_proj_conv(d, np.ascontiguousarray(x["x"][b:b + 1]), x["W"], x["conv_w"], x["conv_b"],
                     x["conv_state"].copy() if decode else x["conv_state"], x["indices"][b:b + 1], write_pool=decode,
                     records=not decode)


def _in_proj_cpu_baseline(w, x, decode: bool, seconds: float) -> dict:
    import oracle

    orc = oracle.default()
    cores = host_cores()
    lanes = [b for b in range(w.B) if x["indices"][b] >= 0]
    work = [(lambda b=b: _in_proj_lane(orc, w, x, b, decode)) for b in lanes]
    done, dt = oracle_throughput(work, seconds, min(cores, max(1, len(work))), cycle=True)
    v = done * w.T / dt
    return {"value": v, "unit": "rows/s", "cores": min(cores, max(1, len(work))), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"the oracle's in_proj + convolution of single lanes of {w.name} (T = {w.T} rows each) over and "
                      f"over for {seconds:g} s, one lane per thread, fp64 C loops; rows/s = lanes done x T / time"}


def run_in_proj_reference_arm(args, name: str, rank: int, world: int):
    """The reference arm of an in_proj workload: the oracle, each step every active lane once (one per thread)."""
    if rank != 0:
        return
    import oracle

    w = IN_PROJ_NAMED[name]()
    decode = name in IN_PROJ_DECODE
    x = w.arrays()
    orc = oracle.default()
    cores = host_cores()
    lanes = [b for b in range(w.B) if x["indices"][b] >= 0]
    t0 = time.perf_counter()
    _in_proj_lane(orc, w, x, lanes[0], decode)
    t_lane = max(time.perf_counter() - t0, 1e-9)
    threads = min(cores, len(lanes))
    n = int(max(1, min(len(lanes), threads * args.ref_seconds / (args.steps + args.warmup) / t_lane)))
    work = [(lambda b=b: _in_proj_lane(orc, w, x, b, decode)) for b in lanes[:n]]
    for _ in range(args.warmup):
        oracle_throughput(work, 1e9, min(threads, n))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_throughput(work, 1e9, min(threads, n))
    dt = time.perf_counter() - t0
    v = n * w.T * args.steps / dt
    desc = (f"each step: the oracle's in_proj + convolution of {n} of the {len(lanes)} active lanes of {w.name}, one "
            f"lane per thread on {min(threads, n)} threads, fp64 C loops; rows/s = lanes x T / time")
    print(json.dumps({
        "impl": "reference", "metric": IN_PROJ_METRIC, "value": v, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": w.name},
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": min(threads, n), "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": desc},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_prefill_reference_arm(args, pw, rank: int, world: int):
    """The reference arm of a prefill workload: the oracle on every host core, each step the first L tokens of
    one (prompt, value head) pair per core, L sized so that warm-up + steps take about --ref-seconds.
    tokens/s = pairs x L / HV / step time."""
    if rank != 0:
        return
    import oracle

    orc = oracle.default()
    x = pw.arrays()
    cores = host_cores()
    pairs = _prefill_pairs(pw, x)
    cu = x["cu_seqlens"]
    b, h = pairs[0]
    n_seq = int(cu[b + 1] - cu[b])
    probe = min(64, n_seq)
    t0 = time.perf_counter()
    _prefill_pair(orc, pw, x, b, h, probe)
    t_tok = max((time.perf_counter() - t0) / probe, 1e-9)
    use = pairs[:cores]
    L = int(max(1, min(min(int(cu[bb + 1] - cu[bb]) for bb, _ in use),
                       args.ref_seconds / (args.steps + args.warmup) / t_tok)))
    work = [(lambda bb=bb, hh=hh: _prefill_pair(orc, pw, x, bb, hh, L)) for bb, hh in use]
    for _ in range(args.warmup):
        oracle_throughput(work, 1e9, len(use))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_throughput(work, 1e9, len(use))
    dt = time.perf_counter() - t0
    v = len(use) * L / pw.HV * args.steps / dt
    desc = (f"each step: oracle prefill of the first {L} tokens of {len(use)} (prompt, value head) pairs of "
            f"{pw.name}, one per thread on {len(use)} threads, fp64 C loops; tokens/s = pairs x L / HV / time")
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": pw.name},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": len(use), "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": desc},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_norm_reference_arm(args, rank: int, world: int, rows: int = 65536 * 32, DV: int = 128):
    """The reference arm of the gated norm: the oracle on the first n rows each step, split over every host
    core, n sized so that warm-up + steps take about --ref-seconds."""
    if rank != 0:
        return
    import oracle

    orc = oracle.default()
    g = W.gated_norm_inputs(rows, DV, "bf16", "bf16", seed=17)
    cores = host_cores()

    def run(lo, hi):
        orc.gated_rmsnorm(g["o"][lo:hi], "bf16", g["z"][lo:hi], "bf16", g["w"], 1e-6)

    t0 = time.perf_counter()
    run(0, 256)
    t_row = max((time.perf_counter() - t0) / 256, 1e-9)
    n = int(max(cores, min(rows, cores * args.ref_seconds / (args.steps + args.warmup) / t_row)))
    cuts = [n * j // cores for j in range(cores + 1)]
    work = [(lambda lo=cuts[j], hi=cuts[j + 1]: run(lo, hi)) for j in range(cores)]
    for _ in range(args.warmup):
        oracle_throughput(work, 1e9, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_throughput(work, 1e9, cores)
    dt = time.perf_counter() - t0
    v = n * args.steps / dt
    desc = (f"each step: oracle gated norm of the first {n} of {rows} rows of DV={DV}, split over {cores} threads, "
            f"fp64 C loops")
    print(json.dumps({
        "impl": "reference", "metric": NORM_METRIC, "value": v, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"gated_rmsnorm_rows{rows}_DV{DV}_bf16"},
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": desc},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---- the oracle as CPU baseline / reference arm -----------------------------------------------------------
def oracle_pairs(w: W.Workload, x: dict, pairs):
    """Per (lane, value head) inputs for the oracle: one lane, one head, its own one-slot pool copy."""
    r = w.HV // w.HK
    out = []
    for b, h in pairs:
        hk = h // r
        slot = int(x["indices"][b])
        y = {
            "q": np.ascontiguousarray(x["q"][b:b + 1, :, hk:hk + 1]),
            "k": np.ascontiguousarray(x["k"][b:b + 1, :, hk:hk + 1]),
            "v": np.ascontiguousarray(x["v"][b:b + 1, :, h:h + 1]),
            "a": np.ascontiguousarray(x["a"][b:b + 1, :, h:h + 1]),
            "b": np.ascontiguousarray(x["b"][b:b + 1, :, h:h + 1]),
            "A_log": np.ascontiguousarray(x["A_log"][h:h + 1]),
            "dt_bias": np.ascontiguousarray(x["dt_bias"][h:h + 1]),
            "pool": np.ascontiguousarray(x["pool"][slot:slot + 1, h:h + 1]),
            "indices": np.zeros(1, np.int32),
            "accept_len": np.ascontiguousarray(x["accept_len"][b:b + 1]),
        }
        out.append(y)
    return out


def oracle_pair_step(orc, w: W.Workload, d: dict, y: dict):
    """The oracle's share of one step for one (lane, head): verify (+ commit), or decode."""
    if w.mode == "decode":
        orc.decode(d, y, y["pool"])
        return
    _, cache, _ = orc.verify(d, y, cache=w.cache)
    if w.commit and w.commit_mode == "replay":
        orc.commit_replay(d, y, y["pool"], y["accept_len"])
    elif w.commit:
        orc.commit(d, y["pool"], y["indices"], cache, y["accept_len"])


def _pair_setup(w: W.Workload):
    import oracle

    orc = oracle.default()
    x = w.arrays()
    d = dict(oracle.dims_of(w), HV=1, HK=1, num_slots=1)
    active = np.flatnonzero(x["indices"] >= 0)
    pairs = [(int(b), h) for b in active for h in range(w.HV)]
    return orc, x, d, pairs


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo, else lscpu, else the machine type)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform

    return platform.machine()


def oracle_throughput(work, seconds: float, threads: int, cycle: bool = False):
    """Runs `work` (callables, one oracle call each) in order on `threads` threads -- each thread takes the next
    item -- until all are done (`cycle`: over and over) or `seconds` have passed; returns (items done,
    elapsed s).  The oracle's ctypes calls release the GIL, so the threads run on separate cores."""
    import itertools

    nxt = itertools.count()
    done = [0] * threads
    t0 = time.perf_counter()
    deadline = t0 + seconds

    def worker(j):
        while time.perf_counter() < deadline:
            i = next(nxt)
            if i >= len(work) and not cycle:
                return
            work[i % len(work)]()
            done[j] += 1

    ts = [threading.Thread(target=worker, args=(j,)) for j in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return sum(done), time.perf_counter() - t0


def _pair_work(orc, w, d, x, pairs):
    return [(lambda y=y: oracle_pair_step(orc, w, d, y)) for y in oracle_pairs(w, x, pairs)]


def cpu_baseline(w: W.Workload, seconds: float):
    """The oracle as it stands (fp64 C loops) on a bounded sample of the workload -- (lane, head) pairs in order
    -- on every host core (the reported value), and on one thread beside it; tokens/s = pairs * T / HV /
    time.  The pairs' inputs are sliced out before the clock starts."""
    orc, x, d, pairs = _pair_setup(w)
    cores = host_cores()
    probe = _pair_work(orc, w, d, x, pairs[:1])[0]
    t0 = time.perf_counter()
    probe()
    t_pair = max(time.perf_counter() - t0, 1e-6)
    one_s, all_s = seconds / 3.0, seconds * 2.0 / 3.0
    n_need = int(min(len(pairs), 1.5 * cores * all_s / t_pair + 1))  # about the work the time allows
    work = _pair_work(orc, w, d, x, pairs[:n_need])
    n1, dt1 = oracle_throughput(work, one_s, 1, cycle=True)
    n, dt = oracle_throughput(work, all_s, cores, cycle=True)
    return {"value": n * w.T / w.HV / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "one_thread": {"value": n1 * w.T / w.HV / dt1, "unit": "tokens/s", "pairs": n1, "seconds": dt1},
            "sample": f"oracle step ({'decode' if w.mode == 'decode' else 'verify+commit'}) of {n} (lane, head) "
                      f"pairs of {w.name} (its first {len(work)} of {len(pairs)} pairs, in order and again), fp64 "
                      f"C loops on {cores} threads (one per core), {dt:.1f} s; one thread: {n1} pairs in "
                      f"{dt1:.1f} s"}


def run_reference_arm(args, w: W.Workload, rank: int, world: int):
    """The reference arm is the oracle on every host core: each step runs a bounded sample of (lane, head)
    pairs, sized so that warm-up + steps take about --ref-seconds in total.  Only rank 0 works."""
    if rank != 0:
        return
    orc, x, d, pairs = _pair_setup(w)
    cores = host_cores()
    probe = _pair_work(orc, w, d, x, pairs[:1])[0]
    t0 = time.perf_counter()
    probe()
    t_pair = max(time.perf_counter() - t0, 1e-6)
    per_step = args.ref_seconds / (args.steps + args.warmup)
    n = int(max(1, min(len(pairs), cores * per_step // t_pair)))
    work = _pair_work(orc, w, d, x, pairs[:n])
    for _ in range(args.warmup):
        oracle_throughput(work, 1e9, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_throughput(work, 1e9, cores)
    dt = time.perf_counter() - t0
    v = n * w.T / w.HV * args.steps / dt
    desc = (f"each step: oracle {'decode' if w.mode == 'decode' else 'verify+commit'} of {n} of {len(pairs)} "
            f"(lane, head) pairs of {w.name}, fp64 C loops on {cores} threads; tokens/s = pairs * T / HV / time")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": w.name},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": desc},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(W.NAMED) + ["sweep", "sweep_replay", "sweep_fused"] + sorted(PREFILL_NAMED)
                    + ["gated_norm"] + sorted(IN_PROJ_NAMED), default="verify4")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--min-seconds", type=float, default=MIN_WINDOW_S,
                    help="minimum device time of each point's timed region (the K steps are repeated to reach it)")
    ap.add_argument("--no-points", action="store_true",
                    help="verify4 line only: leave out the T=1 / T=8 / replay-commit points and the sweep summary")
    ap.add_argument("--sweep-steps", type=int, default=40, help="steps per point of the verify4 line's sweep summary")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if args.workload in IN_PROJ_NAMED:
        if args.impl == "reference":
            run_in_proj_reference_arm(args, args.workload, rank, world)
        else:
            run_in_proj_arm(args, args.workload, rank, world, local_rank)
        return 0
    if args.workload in PREFILL_NAMED or args.workload == "gated_norm":
        if args.impl == "reference":
            if args.workload == "gated_norm":
                run_norm_reference_arm(args, rank, world)
            else:
                run_prefill_reference_arm(args, PREFILL_NAMED[args.workload](), rank, world)
            return 0
        if args.workload == "gated_norm":
            run_norm_arm(args, rank, world, local_rank)
        else:
            run_prefill_arm(args, PREFILL_NAMED[args.workload](), rank, world, local_rank)
        return 0
    if args.workload == "sweep":
        pts = W.sweep()
    elif args.workload == "sweep_replay":
        pts = W.sweep_replay()
    elif args.workload == "sweep_fused":
        pts = W.sweep_fused()
    else:
        pts = [W.NAMED[args.workload]()]
    headline = args.workload == "verify4" and not args.no_points
    for w in pts:
        if args.impl == "reference":
            run_reference_arm(args, w, rank, world)
        else:
            run_cuda_arm(args, w, rank, world, local_rank, points=POINTS if headline else (),
                         sweep_steps=args.sweep_steps if headline else 0)
    return 0


if __name__ == "__main__":
    sys.exit(main())
