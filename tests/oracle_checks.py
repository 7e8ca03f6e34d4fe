"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each ``check_*`` function takes an ``oracle.Oracle`` handle and raises ``AssertionError`` on a mismatch.
``test_oracle_pins.py`` runs them on the committed oracle; ``test_oracle_mutants.py`` runs them on copies of
the oracle with a planted mistake and expects at least one to fail for each mistake.

What pins what:

* bf16 store rounding  -- torch's fp32->bf16 cast (library) on fp32 values; hand-checked ties, overflow and
  a value where rounding through fp32 first would round twice.
* softplus / sigmoid    -- ``numpy.logaddexp(0, x)`` and ``scipy.special.expit`` (library routines).
* gate g                -- closed form exp(-c d) with softplus(a + dt_bias) = c, exp(A_log) = d, through the
  whole recurrence (pure decay after one write).
* beta                  -- read back through the recurrence from a zero state: o = beta v (kh . qh).
* beta = 0              -- pure decay: S_T = (prod g) S_0, o_t = (prod_{s<=t} g_s) S_0 qh_t.
* g = 1, beta = 1 with orthonormal keys -- the delta rule writes v exactly: S kh_s = v_s for every s <= t.
* L2 normalisation eps  -- a query with |q|^2 = eps is scaled by 1/sqrt(2).
* head grouping         -- v-head h reads k-head h // (HV/HK).
* product form          -- an independent dense-matrix NumPy restatement (``oracle/brute.py``), 1e-12.
* chained calls         -- verify(T) == T decodes; cache[t] == state after t+1 decodes; commit(L) == state
  after L decodes == cache[L-1] bit for bit.
* padding / bad data    -- canaries untouched, flag bits set.
* replay commit         -- equals the cached commit bit for bit and the product form after L tokens.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import brute

CANARY = np.float64(-12345.678)


def case(B=1, T=1, HK=1, HV=1, DK=4, DV=4, num_slots=None, qkv="f64", state="f64", seed=0, pool_std=0.3):
    """Dims + arrays in fp64 storage (exact), zero q/k/v/a/b, random pool, distinct slots."""
    num_slots = num_slots or B + 2
    rng = np.random.default_rng(seed)
    d = dict(T=T, HK=HK, HV=HV, DK=DK, DV=DV, num_slots=num_slots, qkv_dtype=qkv, state_dtype=state,
             scale=1.0, l2_eps=1e-6)
    st = {"f64": np.float64, "f32": np.float32}
    x = dict(q=np.zeros((B, T, HK, DK), st[qkv]), k=np.zeros((B, T, HK, DK), st[qkv]),
             v=np.zeros((B, T, HV, DV), st[qkv]), a=np.zeros((B, T, HV), st[qkv]),
             b=np.zeros((B, T, HV), st[qkv]), A_log=np.zeros(HV, np.float32),
             dt_bias=np.zeros(HV, np.float32),
             pool=(rng.standard_normal((num_slots, HV, DV, DK)) * pool_std).astype(st[state]),
             indices=rng.permutation(num_slots)[:B].astype(np.int32))
    return d, x


def rel_err(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-300))


def gate_inputs(c: float, dd: float, dt: float = 0.25):
    """(a, A_log, dt_bias) with softplus(a + dt_bias) = c and exp(A_log) = dd (A_log, dt_bias stored f32)."""
    dt32 = np.float32(dt)
    A32 = np.float32(math.log(dd))
    a = math.log(math.expm1(c)) - float(dt32)
    return a, A32, dt32


# ---------------------------------------------------------------------------------------------------
def check_bf16_rounding(orc):
    import torch

    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * np.exp2(rng.integers(-140, 127, 2000))).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, -1e-41, 2 ** -133, 2 ** -134, 3 * 2 ** -135],
                 np.float32),
    ])
    vals = vals[np.isfinite(vals)]
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.round_bf16(float(v)) for v in vals])
    bad = np.flatnonzero((got != ref) & ~(np.isinf(got) & np.isinf(ref) & (np.sign(got) == np.sign(ref))))
    assert bad.size == 0, f"bf16 rounding differs from torch at {vals[bad[:5]]}: {got[bad[:5]]} vs {ref[bad[:5]]}"
    # ties to even, above-tie from fp64 (no double rounding), overflow
    assert orc.round_bf16(1 + 2 ** -8) == 1.0
    assert orc.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    assert orc.round_bf16(1 + 2 ** -8 + 2 ** -40) == 1 + 2 ** -7
    assert orc.round_bf16(-(1 + 2 ** -8 + 2 ** -40)) == -(1 + 2 ** -7)
    assert orc.round_bf16(255 * 2.0 ** 120) == 255 * 2.0 ** 120
    assert orc.round_bf16(255.49 * 2.0 ** 120) == 255 * 2.0 ** 120
    assert math.isinf(orc.round_bf16(255.5 * 2.0 ** 120))


def check_scalar_functions(orc):
    from scipy.special import expit

    xs = np.concatenate([np.linspace(-40, 40, 401), [-700.0, -1e-9, 0.0, 1e-9, 700.0]])
    for x in xs:
        sp = orc.softplus(x)
        ref = np.logaddexp(0.0, x)
        assert abs(sp - ref) <= 4e-16 * max(1.0, abs(ref)) + 1e-300, (x, sp, ref)
        sg = orc.sigmoid(x)
        assert abs(sg - expit(x)) <= 4e-16 * max(1e-300, expit(x)) + 1e-300, (x, sg, expit(x))
    assert orc.sigmoid(-math.inf) == 0.0 and orc.sigmoid(math.inf) == 1.0
    assert orc.softplus(-math.inf) == 0.0


def check_gate_closed_form(orc):
    """Write v0 along e0 (g=1, beta=1), then one pure-decay token with a chosen gate g = exp(-c d)."""
    for c, dd in [(1.0, math.log(2.0)), (0.5, 2.0), (3.0, 0.1), (2.0, 1.0), (0.05, 16.0), (6.0, 3.0)]:
        d, x = case(T=2, DK=4, DV=3)
        x["pool"][:] = 0.0
        a1, A32, dt32 = gate_inputs(c, dd)
        x["A_log"][0], x["dt_bias"][0] = A32, dt32
        x["k"][0, 0, 0] = [1, 0, 0, 0]
        x["v"][0, 0, 0] = [1.0, -2.0, 0.5]
        x["a"][0, 0, 0] = -np.inf          # softplus(-inf) = 0 -> g = 1
        x["b"][0, 0, 0] = np.inf           # beta = 1
        x["a"][0, 1, 0] = a1
        x["b"][0, 1, 0] = -np.inf          # beta = 0 -> pure decay
        x["q"][0, 1, 0] = [1, 0, 0, 0]
        o, cache, fl = orc.verify(d, x, cache=True)
        assert fl == 0
        unit = 1.0 / (1.0 + 1e-6)          # |kh|^2 and kh . qh for unit vectors
        g_ref = math.exp(-math.exp(float(A32)) * c)
        want = g_ref * np.array([1.0, -2.0, 0.5]) * unit  # S1 = v0 kh0^T; o1 = g S1 qh1
        assert rel_err(o[0, 1, 0], want) < 1e-12, (c, dd, o[0, 1, 0], want)
        assert rel_err(cache[0, 1, 0], g_ref * cache[0, 0, 0]) < 1e-12


def check_beta_sigmoid(orc):
    from scipy.special import expit

    for bval in [-3.0, -0.5, 0.0, 0.7, 4.0]:
        d, x = case(T=1, DK=4, DV=4)
        x["pool"][:] = 0.0
        x["a"][0, 0, 0] = -np.inf
        x["b"][0, 0, 0] = bval
        x["k"][0, 0, 0] = [0, 3, 0, 0]
        x["q"][0, 0, 0] = [0, 3, 0, 0]
        x["v"][0, 0, 0] = [1.0, 2.0, -1.0, 0.25]
        o, _, _ = orc.verify(d, x, cache=False)
        kq = 9.0 / (9.0 + 1e-6)
        beta = o[0, 0, 0] / (x["v"][0, 0, 0] * kq)
        assert np.abs(beta - expit(bval)).max() < 1e-13, (bval, beta, expit(bval))


def check_beta_zero_pure_decay(orc):
    T = 3
    d, x = case(B=2, T=T, HK=1, HV=2, DK=5, DV=3, seed=3)
    softplus_values = [0.7, 2.0, 0.1]       # softplus(a + dt_bias) per token
    x["b"][:] = -np.inf                     # beta = 0
    rng = np.random.default_rng(11)
    x["k"][:] = rng.standard_normal(x["k"].shape)
    x["v"][:] = rng.standard_normal(x["v"].shape)
    for h, dd in enumerate([1.3, 0.2]):     # exp(A_log) per head
        _, A32, dt32 = gate_inputs(1.0, dd, dt=0.25 * (h + 1))
        x["A_log"][h], x["dt_bias"][h] = A32, dt32
        for t, c in enumerate(softplus_values):
            x["a"][:, t, h] = math.log(math.expm1(c)) - float(dt32)
    j = 2
    x["q"][:, :, 0] = 0.0
    x["q"][:, :, 0, j] = 2.0
    o, cache, fl = orc.verify(d, x, cache=True)
    assert fl == 0
    for bi in range(2):
        slot = x["indices"][bi]
        for h in range(2):
            dd_h = math.exp(float(x["A_log"][h]))
            prod = 1.0
            for t, c in enumerate(softplus_values):
                prod *= math.exp(-dd_h * c)
                S_ref = prod * x["pool"][slot, h]
                assert rel_err(cache[bi, t, h], S_ref) < 1e-12
                o_ref = S_ref[:, j] * 2.0 / math.sqrt(4.0 + 1e-6)
                assert rel_err(o[bi, t, h], o_ref) < 1e-12


def check_orthonormal_keys_write_v(orc):
    T, DK, DV = 5, 8, 6
    d, x = case(T=T, DK=DK, DV=DV, seed=5)
    rng = np.random.default_rng(12)
    Q, _ = np.linalg.qr(rng.standard_normal((DK, DK)))
    keys = Q[:, :T].T                       # T orthonormal rows
    x["a"][:] = -np.inf                     # g = 1
    x["b"][:] = np.inf                      # beta = 1
    x["k"][0, :, 0] = keys
    x["q"][0, :, 0] = keys                  # read back the key just written
    x["v"][0, :, 0] = rng.standard_normal((T, DV))
    o, cache, _ = orc.verify(d, x, cache=True)
    kh = keys / math.sqrt(1.0 + 1e-6)
    for t in range(T):
        assert rel_err(o[0, t, 0], x["v"][0, t, 0]) < 1e-5
        for s in range(t + 1):              # earlier writes survive later orthogonal ones
            assert rel_err(cache[0, t, 0] @ kh[s], x["v"][0, s, 0]) < 1e-5


def check_l2norm_eps(orc):
    d, x = case(T=1, DK=4, DV=4, seed=9)
    x["a"][:] = -np.inf
    x["b"][:] = -np.inf                     # g = 1, beta = 0: S unchanged
    alpha = 1e-3                            # alpha^2 = eps
    x["q"][0, 0, 0] = [0, 0, alpha, 0]
    o, _, _ = orc.verify(d, x, cache=False)
    slot = x["indices"][0]
    want = x["pool"][slot, 0][:, 2] / math.sqrt(2.0)
    assert rel_err(o[0, 0, 0], want) < 1e-12


def check_scale(orc):
    d, x = case(B=2, T=2, HK=1, HV=2, DK=8, DV=4, seed=13)
    rng = np.random.default_rng(1)
    for n in ("q", "k", "v", "a", "b"):
        x[n][:] = rng.standard_normal(x[n].shape)
    o1, _, _ = orc.verify(d, x, cache=False)
    d2 = dict(d, scale=0.375)
    o2, _, _ = orc.verify(d2, x, cache=False)
    assert np.array_equal(o2, 0.375 * o1)


def check_head_mapping(orc):
    """HK=2, HV=4: heads 0,1 read k-head 0; heads 2,3 read k-head 1 (all-zero key -> no write)."""
    d, x = case(B=1, T=1, HK=2, HV=4, DK=4, DV=3, seed=17)
    rng = np.random.default_rng(2)
    x["a"][:] = -np.inf
    x["b"][:] = np.inf
    x["k"][0, 0, 0] = rng.standard_normal(4)
    x["k"][0, 0, 1] = 0.0
    x["v"][0, 0] = rng.standard_normal((4, 3))
    x["q"][0, 0] = rng.standard_normal((2, 4))
    _, cache, _ = orc.verify(d, x, cache=True)
    slot = x["indices"][0]
    for h in (2, 3):
        assert np.array_equal(cache[0, 0, h], x["pool"][slot, h]), h
    for h in (0, 1):
        assert not np.allclose(cache[0, 0, h], x["pool"][slot, h]), h


def _random_case(B, T, HK, HV, DK, DV, seed, qkv="f64", state="f64"):
    d, x = case(B=B, T=T, HK=HK, HV=HV, DK=DK, DV=DV, seed=seed, qkv=qkv, state=state)
    rng = np.random.default_rng(seed + 100)
    for n in ("q", "k", "v", "a", "b"):
        x[n][:] = rng.standard_normal(x[n].shape)
    x["A_log"][:] = np.log(rng.uniform(1, 16, HV))
    x["dt_bias"][:] = rng.standard_normal(HV)
    return d, x


def check_product_form(orc):
    import gdn_workloads as W
    import oracle as O

    cases = []
    w = W.tiny()
    cases.append((O.dims_of(w), w.arrays()))
    cases.append(_random_case(B=3, T=4, HK=2, HV=4, DK=8, DV=5, seed=21))
    cases.append(_random_case(B=2, T=3, HK=1, HV=3, DK=16, DV=16, seed=22))
    for d, x in cases:
        dd = dict(d, cache_dtype="f64")
        o, cache, fl = orc.verify(dd, x, cache=True)
        assert fl == 0
        for b in range(x["q"].shape[0]):
            for h in range(d["HV"]):
                ob, states = brute.lane_head(d, x, b, h)
                assert rel_err(o[b, :, h], ob) < 1e-12, (b, h)
                for t, S in enumerate(states):
                    assert rel_err(cache[b, t, h], S) < 1e-12, (b, h, t)


def _slice_token(x, t):
    y = dict(x)
    for n in ("q", "k", "v", "a", "b"):
        y[n] = np.ascontiguousarray(x[n][:, t:t + 1])
    return y


def check_chained_calls(orc):
    """verify(T) == T decodes (o and final state); cache[t] == state after t+1 decodes; commit(L)."""
    T = 4
    d, x = _random_case(B=3, T=T, HK=2, HV=4, DK=8, DV=6, seed=31)
    x["indices"][1] = -1
    o_v, cache, _ = orc.verify(d, x, cache=True)
    pool = x["pool"].copy()
    d1 = dict(d, T=1)
    for t in range(T):
        o_t, _ = orc.decode(d1, _slice_token(x, t), pool)
        for b in (0, 2):
            slot = x["indices"][b]
            assert rel_err(o_t[b, 0], o_v[b, t]) < 1e-13
            assert rel_err(pool[slot], cache[b, t]) < 1e-13
    # commit with accept length L equals the state after L single steps, bit for bit the cache entry
    for L in range(1, T + 1):
        pool_c = x["pool"].copy()
        acc = np.full(3, L, np.int32)
        assert orc.commit(d, pool_c, x["indices"], cache, acc) == 0
        pool_d = x["pool"].copy()
        for t in range(L):
            orc.decode(d1, _slice_token(x, t), pool_d)
        for b in (0, 2):
            slot = x["indices"][b]
            assert np.array_equal(pool_c[slot], cache[b, L - 1])
            assert rel_err(pool_c[slot], pool_d[slot]) < 1e-13
        untouched = np.setdiff1d(np.arange(d["num_slots"]), x["indices"][[0, 2]])
        assert np.array_equal(pool_c[untouched], x["pool"][untouched])


def check_padding_and_bad_data(orc):
    T = 2
    d, x = _random_case(B=4, T=T, HK=1, HV=2, DK=4, DV=4, seed=41)
    num_slots = d["num_slots"]
    x["indices"][:] = [-1, 0, num_slots, -7]            # padded, valid, too large, below -1
    o = np.full((4, T, 2, 4), CANARY)
    cache = np.full((4, T, 2, 4, 4), CANARY)
    o, cache, fl = orc.verify(dict(d, cache_dtype="f64"), x, cache=True, o=o, cache_out=cache)
    assert fl == 1
    for b in (0, 2, 3):
        assert np.all(o[b] == CANARY) and np.all(cache[b] == CANARY)
    assert not np.any(o[1] == CANARY) and not np.any(cache[1] == CANARY)
    pool = x["pool"].copy()
    fl = orc.decode(dict(d, T=T), x, pool)[1]
    assert fl == 1
    assert np.array_equal(np.delete(pool, 0, axis=0), np.delete(x["pool"], 0, axis=0))
    assert not np.array_equal(pool[0], x["pool"][0])
    # commit: padded lane, accept length 0 (no-op), out-of-range accept lengths (flag 2, no-op)
    x["indices"][:] = [-1, 0, 1, 2]
    _, cache, _ = orc.verify(dict(d, cache_dtype="f64"), x, cache=True)
    pool = x["pool"].copy()
    fl = orc.commit(d, pool, x["indices"], cache, np.array([1, 0, T + 1, -1], np.int32))
    assert fl == 2
    assert np.array_equal(pool, x["pool"])


def check_commit_replay(orc):
    """Replay commit == cached commit, bit for bit; == the product-form state after L tokens (brute.py),
    rounded to bf16; accept length 0 is a no-op; lengths outside 0..T set flag 2 and touch nothing."""
    from gdn_workloads import to_bf16_bits

    T = 4
    d, x = _random_case(B=4, T=T, HK=2, HV=4, DK=8, DV=6, seed=51)
    d = dict(d, state_dtype="bf16")
    x["pool"] = to_bf16_bits((np.random.default_rng(52).standard_normal(x["pool"].shape) * 0.2).astype(np.float32))
    x["indices"][2] = -1
    _, cache, _ = orc.verify(d, x, cache=True)
    acc = np.array([1, 3, 2, 4], np.int32)
    p_copy = x["pool"].copy()
    assert orc.commit(d, p_copy, x["indices"], cache, acc) == 0
    p_replay = x["pool"].copy()
    assert orc.commit_replay(d, x, p_replay, acc) == 0
    assert np.array_equal(p_copy, p_replay)
    untouched = np.setdiff1d(np.arange(d["num_slots"]), x["indices"][[0, 1, 3]])
    assert np.array_equal(p_replay[untouched], x["pool"][untouched])
    for b in (0, 1, 3):
        slot = x["indices"][b]
        for h in range(d["HV"]):
            _, states = brute.lane_head(d, x, b, h)
            want = np.array([orc.round_bf16(v) for v in states[acc[b] - 1].ravel()])
            got = brute.decode_storage(p_replay[slot, h], "bf16").ravel()
            assert np.array_equal(got, want), (b, h)
    p_bad = x["pool"].copy()
    assert orc.commit_replay(d, x, p_bad, np.array([0, T + 1, 1, -1], np.int32)) == 2
    assert np.array_equal(p_bad, x["pool"])


ALL_CHECKS = [check_bf16_rounding, check_scalar_functions, check_gate_closed_form, check_beta_sigmoid,
              check_beta_zero_pure_decay, check_orthonormal_keys_write_v, check_l2norm_eps, check_scale,
              check_head_mapping, check_product_form, check_chained_calls, check_padding_and_bad_data,
              check_commit_replay]
