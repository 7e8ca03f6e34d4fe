"""The chunked tensor-core form of gdn_prefill (DK = 64 and 128) against the CPU oracle, through the C ABI.

The form works in chunks of 32 tokens with the state in fp32 for the whole sequence; bf16 q, k, v with DV >= 128
arrive by TMA (raw rows, normalisation as per-token factors), everything else through the token group's own
loads (normalised hi / lo rows), and both ways are covered.  The cases aim at what the form adds over the token
loop: lengths on either side of every chunk boundary (1, 31, 32, 33, 63, 64, 65, 97, 130), a
second block of state rows that is only partly used (DV = 200), sequences of some thousand tokens (error
accumulation over a hundred chunks, fp32 state at the 1e-4 bound), and the decay extremes of the gates: g = 0
(gamma underflows inside the first chunk: every token starts from zero), g = 1 and beta = 0 (pure decay, here no
decay at all: the state must come back unchanged).  Tolerances: see ``gpu_util``.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gdn_workloads as W
from gpu_util import Dev, host, storage_to_f64
from test_gpu_prefill import compare_prefill, run_prefill, small

pytestmark = pytest.mark.gpu


def run_and_compare(pw, x, has_init=True):
    t = Dev(x)
    before = host(t["pool"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = run_prefill(pw, t, err, has_init=has_init)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return compare_prefill(pw, x, host(o), host(t["pool"]), before, has_init=has_init), host(t["pool"])


@pytest.mark.parametrize("DK,qkv,state", [(128, "bf16", "bf16"), (128, "bf16", "f32"), (64, "bf16", "bf16"),
                                          (64, "f32", "bf16"), (64, "f32", "f32"), (128, "f32", "bf16")])
def test_chunk_boundaries(DK, qkv, state):
    lengths = [1, 31, 32, 33, 0, 63, 64, 65, 97, 130]
    pw = small(f"pc_bounds_dk{DK}_{qkv}_{state}", lengths, DK=DK, DV=128, HK=2, HV=4, qkv=qkv, state=state,
               seed=40 + DK, pad=0.1, fresh=0.3)
    run_and_compare(pw, pw.arrays())


def test_second_row_block_ragged():
    pw = small("pc_dv200", [70, 33, 5], DK=128, DV=200, HK=1, HV=2, state="f32", seed=47, fresh=0.34)
    run_and_compare(pw, pw.arrays())


@pytest.mark.parametrize("state", ["f32", "bf16"])
def test_long_sequences(state):
    pw = small(f"pc_long_{state}", [2048, 1531], DK=128, DV=128, HK=1, HV=2, state=state, seed=48, fresh=0.5)
    run_and_compare(pw, pw.arrays())


def _set(x, key, cols, value, dtype):
    a = storage_to_f64(x[key]).astype(np.float32)
    a[:, cols] = value
    x[key] = W._store(a, dtype)


def test_decay_extremes():
    """Head 0: g = 0 (exp(A_log) = 1e4); head 1: g = 1 (exp(A_log) = e^-80); head 2: beta = 0 on every token
    together with g = 1, so its slots come back unchanged; head 3: the ordinary draw."""
    pw = small("pc_decay", [75, 40, 33], DK=128, DV=128, HK=2, HV=4, seed=49, fresh=0.0)
    x = pw.arrays()
    x["A_log"] = x["A_log"].copy()
    x["A_log"][0] = np.float32(np.log(1e4))
    x["A_log"][1] = np.float32(-80.0)
    x["A_log"][2] = np.float32(-80.0)
    _set(x, "b", 2, -200.0, pw.qkv_dtype)
    _, pool_after = run_and_compare(pw, x)
    idx = x["indices"]
    for b in range(pw.B):
        if idx[b] >= 0:
            assert np.array_equal(pool_after[idx[b], 2], x["pool"][idx[b], 2]), "beta = 0, g = 1 changed the state"
