"""Writes ``tiny_oracle.txt``: the oracle's outputs on the tiny workload (B=2, 4 slots, HK=HV=2, DK=DV=16,
T=2, fp32, seed 0), for regression of the oracle itself.

The pages print no worked example for the gated delta rule, so no value here comes from them; every value
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


if __name__ == "__main__":
    main()
