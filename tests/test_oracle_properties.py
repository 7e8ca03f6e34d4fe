"""Property tests of the CPU oracle (hypothesis): on randomly drawn small shapes, storage types and prompt
mixes, the loop oracle (``gdn_oracle.c``) agrees with the independent NumPy product form (``oracle/brute.py``),
for verify (every token's o and state) and for prefill (every prompt's o and final state, fresh or from its
slot).  This widens the fixed cases of ``oracle_checks.check_product_form`` and
``check_prefill_product_form`` to shapes nobody picked by hand."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import brute  # noqa: E402
from oracle_checks import rel_err  # noqa: E402

STORE = {"f64": np.float64, "f32": np.float32}


def draw_inputs(rng, HK, HV, DK, DV, num_slots, qkv, state, lead):
    f = STORE[qkv]
    return dict(q=rng.standard_normal(lead + (HK, DK)).astype(f), k=rng.standard_normal(lead + (HK, DK)).astype(f),
                v=rng.standard_normal(lead + (HV, DV)).astype(f), a=rng.standard_normal(lead + (HV,)).astype(f),
                b=rng.standard_normal(lead + (HV,)).astype(f),
                A_log=np.log(rng.uniform(1, 16, HV)).astype(np.float32),
                dt_bias=rng.standard_normal(HV).astype(np.float32),
                pool=(rng.standard_normal((num_slots, HV, DV, DK)) * 0.3).astype(STORE[state]))


shapes = st.tuples(st.integers(1, 3),            # HK
                   st.integers(1, 3),            # HV / HK
                   st.sampled_from([1, 2, 5, 8]),  # DK
                   st.integers(1, 6),            # DV
                   st.sampled_from(["f64", "f32"]),
                   st.sampled_from(["f64", "f32"]),
                   st.integers(0, 2 ** 31 - 1))


@settings(max_examples=40, deadline=None)
@given(shapes, st.integers(1, 3), st.integers(1, 5))
def test_verify_matches_product_form(shape, B, T):
    HK, r, DK, DV, qkv, state, seed = shape
    HV = HK * r
    rng = np.random.default_rng(seed)
    num_slots = B + 2
    x = draw_inputs(rng, HK, HV, DK, DV, num_slots, qkv, state, (B, T))
    x["indices"] = rng.permutation(num_slots)[:B].astype(np.int32)
    d = dict(T=T, HK=HK, HV=HV, DK=DK, DV=DV, num_slots=num_slots, qkv_dtype=qkv, state_dtype=state,
             cache_dtype="f64", scale=1.0, l2_eps=1e-6)
    o, cache, fl = oracle.default().verify(d, x, cache=True)
    assert fl == 0
    for b in range(B):
        for h in range(HV):
            ob, states = brute.lane_head(d, x, b, h)
            assert rel_err(o[b, :, h], ob) < 1e-11
            for t, S in enumerate(states):
                assert rel_err(cache[b, t, h], S) < 1e-11


@settings(max_examples=40, deadline=None)
@given(shapes, st.lists(st.integers(0, 9), min_size=1, max_size=4), st.data())
def test_prefill_matches_product_form(shape, lengths, data):
    HK, r, DK, DV, qkv, state, seed = shape
    HV = HK * r
    rng = np.random.default_rng(seed)
    B = len(lengths)
    N = sum(lengths)
    num_slots = B + 2
    x = draw_inputs(rng, HK, HV, DK, DV, num_slots, qkv, state, (N,))
    x["indices"] = rng.permutation(num_slots)[:B].astype(np.int32)
    init = np.array(data.draw(st.lists(st.integers(0, 1), min_size=B, max_size=B)), np.int32)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    d = dict(T=N, HK=HK, HV=HV, DK=DK, DV=DV, num_slots=num_slots, qkv_dtype=qkv, state_dtype=state,
             scale=1.0, l2_eps=1e-6)
    pool = x["pool"].copy()
    o, fl = oracle.default().prefill(d, x, cu, pool, init)
    assert fl == 0
    for b in range(B):
        if lengths[b] == 0:
            assert np.array_equal(pool[x["indices"][b]], x["pool"][x["indices"][b]])
            continue
        for h in range(HV):
            ob, S = brute.sequence_head(d, x, cu, init, b, h)
            assert rel_err(o[cu[b]:cu[b + 1], h], ob) < 1e-11
            if state == "f64":
                assert rel_err(pool[x["indices"][b], h], S) < 1e-11
            else:  # stored once, rounded to fp32
                assert np.abs(pool[x["indices"][b], h] - S).max() <= 1e-6 * max(np.abs(S).max(), 1e-30)
