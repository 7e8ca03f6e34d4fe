"""Width transitions on one pool: calls of different T in a row -- T = 8, 1, 3, 2, 8, 4 -- each verify followed
by its commit (the copy commit after a caching verify, the replay commit after a verify without intermediate
states; T = 1 is a decode).  The sequence crosses every kernel of the launcher (direct, bulk-copy staged,
chunked) and the chunked kernel's per-T launch caches, on one pool that each step leaves to the next.

Every step is checked against the oracle run from the pool exactly as the GPU left it before that step, so
each step gets the tolerances of a single call and a difference cannot carry over.  Slots of padded lanes
and unreferenced slots stay bitwise unchanged throughout.  Tolerances: see ``gpu_util``.  The sequence takes
its calls from a backend object, so that the same steps can run against an oracle-backed stand-in on a CPU
to check the test itself.
"""
from __future__ import annotations

import numpy as np
import pytest

import gdn_workloads as W
import oracle

pytestmark = pytest.mark.gpu

# (T, step kind); "cache": verify with intermediate states + gdn_commit, "replay": verify without them +
# gdn_commit_replay, "decode": gdn_decode
STEPS = [(8, "cache"), (1, "decode"), (3, "replay"), (2, "cache"), (8, "replay"), (4, "cache")]


def base_workload() -> W.Workload:
    # 16 lanes x 32 value heads: enough CTAs for the staged kernel at T <= 2; one padded lane
    return W.Workload("transitions", B=16, T=1, HK=16, HV=32, DK=128, DV=128, num_slots=24, qkv_dtype="bf16",
                      state_dtype="bf16", out_dtype="bf16", mode="verify", cache=True, commit=True, seed=61,
                      pool_std=0.1, pad_fraction=0.07)


def step_inputs(w0: W.Workload, i: int, T: int) -> dict:
    """Fresh tokens and accept lengths for step i; the lanes (slots) and the per-head A_log, dt_bias stay."""
    first = w0.small_arrays()
    x = w0.replace(T=T, seed=w0.seed + 101 * (i + 1)).small_arrays()
    for k in ("indices", "A_log", "dt_bias"):
        x[k] = first[k]
    return x


def run_transitions(backend) -> None:
    """The sequence, with `backend` doing the calls: to_dev(dict) -> device dict, host(t) -> storage array,
    verify(w, t, pool, cache) -> (o, cache or None), commit(pool, idx, cache, acc), replay(w, t, pool, acc),
    decode(w, t, pool) -> o, and checks check_o(w, got, ref, what), check_state(w, got, ref, what)."""
    w0 = base_workload()
    orc = oracle.default()
    pool = backend.to_dev({"pool": w0.pool()})["pool"]
    first = w0.small_arrays()
    active = first["indices"][first["indices"] >= 0]
    assert len(active) < w0.B  # at least one padded lane
    untouched = np.setdiff1d(np.arange(w0.num_slots), active)
    start = backend.host(pool)
    for i, (T, kind) in enumerate(STEPS):
        w = w0.replace(T=T, mode="decode" if kind == "decode" else "verify", cache=kind == "cache")
        x = step_inputs(w0, i, T)
        before = backend.host(pool)
        xr = dict(x, pool=before.copy())
        t = backend.to_dev(x)
        d = oracle.dims_of(w)
        what = f"step {i} (T={T}, {kind})"
        if kind == "decode":
            o = backend.decode(w, t, pool)
            o_ref, fl = orc.decode(d, xr, xr["pool"])
        else:
            o, cache = backend.verify(w, t, pool, kind == "cache")
            o_ref, c_ref, fl = orc.verify(d, xr, cache=kind == "cache")
            if kind == "cache":
                backend.check_state(w, backend.host(cache)[x["indices"] >= 0], c_ref[x["indices"] >= 0],
                                    what + " intermediate states")
                backend.commit(pool, t["indices"], cache, t["accept_len"])
                assert orc.commit(d, xr["pool"], x["indices"], c_ref, x["accept_len"]) == 0
            else:
                backend.replay(w, t, pool, t["accept_len"])
                assert orc.commit_replay(d, xr, xr["pool"], x["accept_len"]) == 0
        assert fl == 0
        act = x["indices"] >= 0
        backend.check_o(w, backend.host(o)[act], o_ref[act], what + " o")
        after = backend.host(pool)
        backend.check_state(w, after[active], xr["pool"][active], what + " pool")
        assert np.array_equal(after[untouched], start[untouched]), what + ": an unreferenced slot changed"


class GpuBackend:
    """The library through its binding on cuda:0."""

    def __init__(self):
        import torch

        import gated_deltanet_linear_mtp_gb300 as gdn
        import gpu_util as G

        self.torch, self.gdn, self.G = torch, gdn, G
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def to_dev(self, x):
        return {k: self.G.dev(v) for k, v in x.items()}

    def host(self, t):
        self.torch.cuda.synchronize()
        assert int(self.err.item()) == 0, f"device error word {int(self.err.item())}"
        return self.G.host(t)

    def verify(self, w, t, pool, cache):
        return self.G.run_verify(w, dict(t, pool=pool), cache=cache, err=self.err)

    def commit(self, pool, idx, cache, acc):
        self.gdn.gdn_commit(pool, idx, cache, acc, self.err)

    def replay(self, w, t, pool, acc):
        self.gdn.gdn_commit_replay(t["q"], t["k"], t["v"], t["a"], t["b"], t["A_log"], t["dt_bias"], pool,
                                   t["indices"], acc, self.err, scale=w.scale, l2_eps=w.l2_eps)

    def decode(self, w, t, pool):
        return self.G.run_decode(w, t, pool, err=self.err)

    def check_o(self, w, got, ref, what):
        self.G.check_o(w, got, ref, what)

    def check_state(self, w, got, ref, what):
        self.G.check_state(w, got, ref, what)


def test_width_transitions_each_followed_by_commit():
    run_transitions(GpuBackend())
    run_transitions(GpuBackend())  # again, with every launch cache already filled
