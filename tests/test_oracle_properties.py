"""Property tests of the CPU oracle (hypothesis): on randomly drawn small shapes, storage types and prompt
mixes, the loop oracle (``gdn_oracle.c``) agrees with the independent NumPy product form (``oracle/brute.py``),
for verify (every token's o and state) and for prefill (every prompt's o and final state, fresh or from its
slot); and the in_proj + conv1d against a NumPy restatement.  This widens the fixed cases of
``oracle_checks.check_product_form``, ``check_prefill_product_form`` and ``check_conv_is_numpy_convolve`` to
shapes nobody picked by hand."""
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


@settings(max_examples=40, deadline=None)
@given(st.tuples(st.integers(1, 2), st.integers(1, 2), st.integers(1, 4), st.integers(1, 5), st.integers(1, 9),
                 st.integers(1, 4), st.integers(1, 5), st.integers(1, 3), st.sampled_from(["f64", "f32"]),
                 st.booleans(), st.integers(0, 2 ** 31 - 1)))
def test_in_proj_conv_matches_numpy(case):
    """The in_proj projection with its causal conv1d: the loop oracle against a NumPy restatement (matrix product,
    then numpy.convolve per channel over [state, rows] with the taps reversed, scipy's expit), on random shapes,
    tap counts, state types and SiLU on or off; the written-back state is the sequence's last K - 1 entries."""
    from scipy.special import expit

    HK, r, DK, DV, H, K, T, B, conv, silu, seed = case
    HV = HK * r
    rng = np.random.default_rng(seed)
    num_slots = B + 2
    Cc = 2 * HK * DK + HV * DV
    C = Cc + HV * DV + 2 * HV
    x = rng.standard_normal((B, T, H))
    Wm = rng.standard_normal((C, H))
    taps = rng.uniform(-1, 1, (Cc, K)).astype(np.float32)
    bias = rng.normal(0, 0.3, Cc).astype(np.float32)
    pool = rng.standard_normal((num_slots, K - 1, Cc)).astype(STORE[conv])
    idx = rng.permutation(num_slots)[:B].astype(np.int32)
    d = dict(T=T, H=H, HK=HK, HV=HV, DK=DK, DV=DV, K=K, num_slots=num_slots, x_dtype="f64", conv_dtype=conv,
             silu=int(silu))
    before = pool.copy()
    out, rec, fl = oracle.default().in_proj_conv(d, x, Wm, taps, bias, pool, idx, write_pool=True)
    assert fl == 0
    p = np.einsum("ch,bth->btc", Wm, x)  # another summation order: equal up to the last fp64 bits
    assert rel_err(out[..., Cc:], p[..., Cc:]) <= 1e-12
    u = rec.astype(np.float64)  # the values the state stores: the product rounded once to the state's type
    step = 1e-12 if conv == "f64" else 2.0 ** -23
    assert np.all(np.abs(u - p[..., :Cc]) <= step * np.abs(p[..., :Cc]) + 1e-300)
    for b in range(B):
        for c in range(Cc):
            seq = np.concatenate([before[idx[b], :, c].astype(np.float64), u[b, :, c]])
            y = float(bias[c]) + np.convolve(seq, taps[c, ::-1].astype(np.float64), mode="valid")
            if silu:
                y = y * expit(y)
            assert np.abs(out[b, :, c] - y).max() <= 1e-12 * max(1.0, np.abs(y).max()), (b, c)
            assert np.array_equal(pool[idx[b], :, c].astype(np.float64), seq[T:]), (b, c)
