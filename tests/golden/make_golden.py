"""Writes ``tiny_oracle.txt``: the oracle's outputs on the tiny workload (B=2, 4 slots, HK=HV=2, DK=DV=16,
T=2, fp32, seed 0), and ``tiny_in_proj_oracle.txt``: its in_proj + conv1d on a tiny projection, for regression of
the oracle itself.

The pages print no worked example for the gated delta rule or the projection, so no value here comes from them; every value
is written by this script, which calls only ``oracle/`` and the seeded input generator.  Run from the repo
root: ``python tests/golden/make_golden.py``.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import gdn_workloads as W  # noqa: E402
import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.txt")
OUT_IN_PROJ = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_in_proj_oracle.txt")


def in_proj_workload():
    """B=2 lanes x T=3 rows of H=16, HK=1, HV=2, DK=DV=4 (C = 28, Cc = 16), K=4 taps, fp32 state and outputs,
    4 slots, seed 7."""
    return W.InProjWorkload("tiny_in_proj", B=2, T=3, H=16, HK=1, HV=2, DK=4, DV=4, K=4, num_slots=4,
                            conv_dtype="f32", out_dtype="f32", seed=7)


def compute_in_proj():
    """The oracle's in_proj + conv1d on the tiny workload: verify rows (outputs and records), then decode rows from
    the same state (the written-back state)."""
    w = in_proj_workload()
    x = w.arrays()
    d = dict(T=w.T, H=w.H, HK=w.HK, HV=w.HV, DK=w.DK, DV=w.DV, K=w.K, num_slots=w.num_slots, x_dtype="bf16",
             conv_dtype="f32", silu=1)
    orc = oracle.default()
    out, rec, fl = orc.in_proj_conv(d, x["x"], x["W"], x["conv_w"], x["conv_b"], x["conv_state"], x["indices"],
                                    write_pool=False)
    assert fl == 0
    state = x["conv_state"].copy()
    assert orc.in_proj_conv(d, x["x"], x["W"], x["conv_w"], x["conv_b"], state, x["indices"], write_pool=True,
                            records=False)[2] == 0
    return dict(indices=x["indices"], out=out.ravel(), rec_bits=rec.view(np.uint32).ravel(),
                state_bits=state.view(np.uint32).ravel())


def compute():
    w = W.tiny()
    x = w.arrays()
    d = oracle.dims_of(w)
    orc = oracle.default()
    o, cache, fl = orc.verify(d, x, cache=True)
    assert fl == 0
    pool = x["pool"].copy()
    assert orc.commit(d, pool, x["indices"], cache, x["accept_len"]) == 0
    return dict(o=o.ravel(), cache_bits=cache.view(np.uint32).ravel(), pool_bits=pool.view(np.uint32).ravel(),
                accept_len=x["accept_len"], indices=x["indices"])


def main():
    r = compute()
    with open(OUT, "w") as f:
        f.write("# oracle outputs on the tiny fp32 workload (seed 0); written by tests/golden/make_golden.py\n")
        f.write("# o: fp64 hex floats [B,T,HV,DV]; cache_bits / pool_bits: fp32 bit patterns (hex)\n")
        f.write("indices " + " ".join(str(int(v)) for v in r["indices"]) + "\n")
        f.write("accept_len " + " ".join(str(int(v)) for v in r["accept_len"]) + "\n")
        f.write("o " + " ".join(float(v).hex() for v in r["o"]) + "\n")
        f.write("cache_bits " + " ".join(f"{int(v):08x}" for v in r["cache_bits"]) + "\n")
        f.write("pool_bits " + " ".join(f"{int(v):08x}" for v in r["pool_bits"]) + "\n")


    r = compute_in_proj()
    with open(OUT_IN_PROJ, "w") as f:
        f.write("# oracle in_proj + conv1d on the tiny workload of in_proj_workload(); written by tests/golden/make_golden.py\n")
        f.write("# out: fp64 hex floats [B,T,C]; rec_bits / state_bits: fp32 bit patterns (hex)\n")
        f.write("indices " + " ".join(str(int(v)) for v in r["indices"]) + "\n")
        f.write("out " + " ".join(float(v).hex() for v in r["out"]) + "\n")
        f.write("rec_bits " + " ".join(f"{int(v):08x}" for v in r["rec_bits"]) + "\n")
        f.write("state_bits " + " ".join(f"{int(v):08x}" for v in r["state_bits"]) + "\n")


if __name__ == "__main__":
    main()
