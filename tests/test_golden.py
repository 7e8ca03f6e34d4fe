"""The oracle reproduces its stored outputs on the tiny workloads (``tests/golden/tiny_oracle.txt``,
``tests/golden/tiny_in_proj_oracle.txt``)."""
import os

import numpy as np

from golden import make_golden


def _load(path=None):
    rows = {}
    with open(path or make_golden.OUT) as f:
        for line in f:
            if line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = vals
    return rows


def test_tiny_golden():
    g = _load()
    r = make_golden.compute()
    assert [int(v) for v in g["indices"]] == list(r["indices"])
    assert [int(v) for v in g["accept_len"]] == list(r["accept_len"])
    o_ref = np.array([float.fromhex(v) for v in g["o"]])
    # libm's exp/log1p may differ in the last bit between machines: 1e-14 relative
    assert np.abs(r["o"] - o_ref).max() <= 1e-14 * np.abs(o_ref).max()
    cache_ref = np.array([int(v, 16) for v in g["cache_bits"]], np.uint32).view(np.float32)
    pool_ref = np.array([int(v, 16) for v in g["pool_bits"]], np.uint32).view(np.float32)
    cache = r["cache_bits"].view(np.float32)
    pool = r["pool_bits"].view(np.float32)
    assert np.abs(cache - cache_ref).max() <= 1e-6 * np.abs(cache_ref).max()
    assert np.abs(pool - pool_ref).max() <= 1e-6 * np.abs(pool_ref).max()


def test_tiny_in_proj_golden():
    g = _load(make_golden.OUT_IN_PROJ)
    r = make_golden.compute_in_proj()
    assert [int(v) for v in g["indices"]] == list(r["indices"])
    out_ref = np.array([float.fromhex(v) for v in g["out"]])
    # SiLU's exp may differ in the last bit between machines' libm: 1e-14 relative
    assert np.abs(r["out"] - out_ref).max() <= 1e-14 * np.abs(out_ref).max()
    for key in ("rec_bits", "state_bits"):  # stored products (no libm): identical
        assert np.array_equal(np.array([int(v, 16) for v in g[key]], np.uint32), r[key]), key
