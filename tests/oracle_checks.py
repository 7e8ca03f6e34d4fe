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


def _prefill_case(lengths, HK=2, HV=4, DK=8, DV=6, seed=61, qkv="f64", state="f64"):
    """Packed prefill inputs for sequences of the given lengths (random q, k, v, a, b, gates, pool)."""
    N = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    B = len(lengths)
    rng = np.random.default_rng(seed)
    st = {"f64": np.float64, "f32": np.float32}
    num_slots = B + 3
    d = dict(T=N, HK=HK, HV=HV, DK=DK, DV=DV, num_slots=num_slots, qkv_dtype=qkv, state_dtype=state,
             scale=1.0, l2_eps=1e-6)
    x = dict(q=rng.standard_normal((N, HK, DK)).astype(st[qkv]), k=rng.standard_normal((N, HK, DK)).astype(st[qkv]),
             v=rng.standard_normal((N, HV, DV)).astype(st[qkv]), a=rng.standard_normal((N, HV)).astype(st[qkv]),
             b=rng.standard_normal((N, HV)).astype(st[qkv]),
             A_log=np.log(rng.uniform(1, 16, HV)).astype(np.float32),
             dt_bias=rng.standard_normal(HV).astype(np.float32),
             pool=(rng.standard_normal((num_slots, HV, DV, DK)) * 0.3).astype(st[state]),
             indices=rng.permutation(num_slots)[:B].astype(np.int32))
    return d, x, cu


def check_prefill_product_form(orc):
    """Variable-length sequences, with and without an initial state, against the product form
    (brute.sequence_head); a padded sequence and an empty one leave o and the pool as they were."""
    lengths = [5, 1, 0, 7, 3, 4]
    d, x, cu = _prefill_case(lengths)
    x["indices"][4] = -1
    init = np.array([1, 0, 1, 0, 1, 1], np.int32)
    pool = x["pool"].copy()
    o0 = np.full((cu[-1], d["HV"], d["DV"]), CANARY)
    o, fl = orc.prefill(d, x, cu, pool, init, o=o0.copy())
    assert fl == 0
    for b in range(len(lengths)):
        lo, hi = cu[b], cu[b + 1]
        slot = x["indices"][b]
        if slot < 0:
            assert np.all(o[lo:hi] == CANARY)
            continue
        if lengths[b] == 0:
            assert np.array_equal(pool[slot], x["pool"][slot])
            continue
        for h in range(d["HV"]):
            ob, S = brute.sequence_head(d, x, cu, init, b, h)
            assert rel_err(o[lo:hi, h], ob) < 1e-12, (b, h)
            assert rel_err(pool[slot, h], S) < 1e-12, (b, h)
    touched = x["indices"][[0, 1, 3, 5]]
    untouched = np.setdiff1d(np.arange(d["num_slots"]), touched)
    assert np.array_equal(pool[untouched], x["pool"][untouched])


def check_prefill_fresh_state(orc):
    """A sequence without an initial state never reads its slot (NaN there changes nothing) and starts from
    zero: after one token S = beta v kh^T, so o = beta v (kh . qh)."""
    from scipy.special import expit

    d, x, cu = _prefill_case([1, 3], HK=1, HV=2, DK=4, DV=3, seed=62)
    init = np.array([0, 0], np.int32)
    pool = x["pool"].copy()
    pool[x["indices"]] = np.nan
    o, fl = orc.prefill(d, x, cu, pool, init)
    assert fl == 0 and np.all(np.isfinite(o)) and np.all(np.isfinite(pool[x["indices"]]))
    pool_zero = x["pool"].copy()
    pool_zero[x["indices"]] = 0.0
    o2, _ = orc.prefill(d, x, cu, pool_zero, np.array([1, 1], np.int32))
    assert np.array_equal(o, o2) and np.array_equal(pool[x["indices"]], pool_zero[x["indices"]])
    for h in range(2):
        q, k, v = x["q"][0, 0], x["k"][0, 0], x["v"][0, h]
        kq = (k @ q) / math.sqrt((k @ k + 1e-6) * (q @ q + 1e-6))
        want = expit(float(x["b"][0, h])) * v * kq
        assert rel_err(o[0, h], want) < 1e-12, h


def check_prefill_matches_verify_and_decode(orc):
    """Equal lengths T packed lane after lane are the [B, T] layout of verify: same outputs as verify, and
    the final state written back is the one decode(T) writes."""
    T, B = 3, 3
    d, x, cu = _prefill_case([T] * B, HK=2, HV=4, DK=8, DV=5, seed=63)
    x["indices"][1] = -1
    pool = x["pool"].copy()
    o, fl = orc.prefill(d, x, cu, pool)
    assert fl == 0
    dv = dict(d, T=T)
    xv = dict(x)
    for n, shape in (("q", (B, T, d["HK"], d["DK"])), ("k", (B, T, d["HK"], d["DK"])),
                     ("v", (B, T, d["HV"], d["DV"])), ("a", (B, T, d["HV"])), ("b", (B, T, d["HV"]))):
        xv[n] = np.ascontiguousarray(x[n].reshape(shape))
    o_v, _, _ = orc.verify(dv, xv, cache=False)
    pool_d = x["pool"].copy()
    orc.decode(dv, xv, pool_d)
    for b in (0, 2):
        assert np.array_equal(o[b * T:(b + 1) * T], o_v[b])
    assert np.array_equal(pool, pool_d)


def check_prefill_chained(orc):
    """A sequence split in two prefill calls (the second from the state the first wrote) equals one call."""
    d, x, cu = _prefill_case([9], HK=1, HV=2, DK=8, DV=4, seed=64)
    pool_one = x["pool"].copy()
    o_one, _ = orc.prefill(d, x, cu, pool_one)
    for L1 in (1, 4, 8):
        pool = x["pool"].copy()
        x1 = dict(x, **{n: np.ascontiguousarray(x[n][:L1]) for n in ("q", "k", "v", "a", "b")})
        x2 = dict(x, **{n: np.ascontiguousarray(x[n][L1:]) for n in ("q", "k", "v", "a", "b")})
        o1, _ = orc.prefill(dict(d, T=L1), x1, np.array([0, L1], np.int32), pool, np.ones(1, np.int32))
        o2, _ = orc.prefill(dict(d, T=9 - L1), x2, np.array([0, 9 - L1], np.int32), pool)
        assert rel_err(np.concatenate([o1, o2]), o_one) < 1e-13, L1
        assert rel_err(pool, pool_one) < 1e-13, L1


def check_prefill_bad_bounds(orc):
    """Decreasing, negative or too-long sequence bounds skip the sequence and set flag 8; an out-of-range
    index flag 1; nothing is written for them."""
    d, x, cu = _prefill_case([2, 3], HK=1, HV=1, DK=4, DV=4, seed=65)
    for bad in ([0, 3, 2], [-1, 2, 5], [0, 2, 6]):
        pool = x["pool"].copy()
        o, fl = orc.prefill(d, x, np.array(bad, np.int32), pool, o=np.full((5, 1, 4), CANARY))
        assert fl == 8, (bad, fl)
        ok = [b for b in range(2) if 0 <= bad[b] <= bad[b + 1] <= 5]
        for b in range(2):
            if b not in ok:
                assert np.array_equal(pool[x["indices"][b]], x["pool"][x["indices"][b]]), bad
    x["indices"][0] = d["num_slots"]
    pool = x["pool"].copy()
    o, fl = orc.prefill(d, x, cu, pool, o=np.full((5, 1, 4), CANARY))
    assert fl == 1 and np.all(o[0:2] == CANARY) and not np.any(o[2:5] == CANARY)


def check_gated_rmsnorm_closed_forms(orc):
    """Rows with a closed-form RMS (one-hot, constant, a 3-4-5 pair, zero) and gates z = ln r, where
    silu(ln r) = ln r * r / (1 + r) exactly; weights differ per column, gates per row and column."""
    DV = 4
    w = np.array([0.5, -2.0, 1.25, 3.0], np.float32)
    r = np.array([[3.0, 0.25, 7.0, 1.5], [2.0, 9.0, 0.5, 4.0], [5.0, 0.2, 1.0, 6.0], [1.25, 3.0, 8.0, 0.75],
                  [4.0, 4.0, 0.1, 2.5]])
    z = np.log(r)
    silu = np.log(r) * r / (1.0 + r)
    for eps in (0.0, 1e-6, 0.75):
        o = np.array([[0.0, 2.5, 0.0, 0.0],       # one-hot: mean = c^2 / DV
                      [-1.5, -1.5, -1.5, -1.5],   # constant
                      [3.0, 0.0, 4.0, 0.0],       # mean = 25 / 4
                      [0.0, 0.0, 0.0, 0.0],       # zero row
                      [1.0, -1.0, 1.0, -1.0]])
        rms = np.sqrt(np.array([2.5 ** 2 / DV, 2.25, 25.0 / 4, 0.0, 1.0]) + eps)
        y = orc.gated_rmsnorm(o, "f64", z, "f64", w, eps)
        for i in range(5):
            if i == 3 and eps == 0.0:
                continue                          # 0 / 0: no closed form
            want = o[i] / rms[i] * w.astype(np.float64) * silu[i]
            assert np.abs(y[i] - want).max() <= 1e-14 * max(1.0, np.abs(want).max()), (eps, i, y[i], want)
    # storage types are read exactly: bf16 o and z (bit patterns), fp32 rows
    from gdn_workloads import to_bf16_bits
    ob = to_bf16_bits(np.array([[3.0, 0.0, 4.0, 0.0]], np.float32))
    zb = to_bf16_bits(np.array([[1.0, 2.0, -1.0, 0.5]], np.float32))
    y = orc.gated_rmsnorm(ob, "bf16", zb, "bf16", w, 0.0)
    zz = np.array([1.0, 2.0, -1.0, 0.5])
    want = np.array([3.0, 0.0, 4.0, 0.0]) / 2.5 * w * (zz / (1 + np.exp(-zz)))
    assert np.abs(y[0] - want).max() < 1e-14


# ---- the in_proj projection with its causal conv1d epilogue -------------------------------------------------
def _conv_case(B=2, T=3, H=5, HK=1, HV=2, DK=2, DV=3, K=4, x="f64", conv="f64", silu=1, seed=70, identity=False):
    """Dims and fp64-exact arrays: x ~ N(0,1), W ~ N(0, 1/H) (or the identity with H = C), conv taps U(-1, 1)
    and biases in fp32, a random convolution-state pool, distinct random slots."""
    import oracle

    num_slots = B + 2
    rng = np.random.default_rng(seed)
    d = dict(T=T, H=H, HK=HK, HV=HV, DK=DK, DV=DV, K=K, num_slots=num_slots, x_dtype=x, conv_dtype=conv, silu=silu)
    Cc, C = oracle.conv_channels(d)
    if identity:
        d["H"] = H = C
    xs = rng.normal(size=(B, T, H))
    Wm = np.eye(C) if identity else rng.normal(size=(C, H)) / math.sqrt(H)
    conv_w = rng.uniform(-1.0, 1.0, (Cc, K)).astype(np.float32)
    conv_b = rng.normal(0.0, 0.3, Cc).astype(np.float32)
    pool = rng.normal(size=(num_slots, K - 1, Cc))
    if conv == "f32":
        pool = pool.astype(np.float32)
    idx = rng.permutation(num_slots)[:B].astype(np.int32)
    if x == "f32":
        xs, Wm = xs.astype(np.float32), Wm.astype(np.float32)
    return d, xs, Wm, conv_w, conv_b, pool, idx


def check_in_proj_is_the_matrix_product(orc):
    """With the current-row tap alone (w = e_{K-1}), no bias and no SiLU, every output channel is the product
    W x of the row (numpy's matmul), the recovery records hold the same for q, k, v, and the pool is read only."""
    import oracle

    for K in (1, 2, 4):
        d, xs, Wm, _, _, pool, idx = _conv_case(K=K, silu=0, seed=71 + K)
        Cc, C = oracle.conv_channels(d)
        taps = np.zeros((Cc, K), np.float32)
        taps[:, K - 1] = 1.0
        before = pool.copy()
        out, rec, fl = orc.in_proj_conv(d, xs, Wm, taps, None, pool, idx, write_pool=False)
        want = np.einsum("ch,bth->btc", Wm, xs)
        assert fl == 0
        assert np.abs(out - want).max() <= 1e-12 * np.abs(want).max(), K
        assert np.abs(rec - want[..., :Cc]).max() <= 1e-12 * np.abs(want).max(), K
        assert np.array_equal(pool, before)
        parts = oracle.split_in_proj(d, want)
        assert parts["q"].shape == (2, 3, 1, 2) and parts["z"].shape == (2, 3, 2, 3) and parts["a"].shape == (2, 3, 2)
        assert np.array_equal(parts["a"], want[..., -2:]) and np.array_equal(parts["v"].reshape(2, 3, 6), want[..., 4:10])


def check_conv_is_numpy_convolve(orc):
    """W = I (p = x): each convolved channel is bias + the 'valid' correlation of [state, x rows] with its taps
    (numpy.convolve with the taps reversed), SiLU by scipy's expit; the decode write-back keeps the last K-1
    entries of that sequence; the other channels pass x through."""
    import oracle
    from scipy.special import expit

    for K, T, silu in ((4, 3, 0), (4, 1, 1), (2, 5, 1), (3, 2, 0)):
        d, xs, Wm, taps, bias, pool, idx = _conv_case(K=K, T=T, silu=silu, seed=80 + K + T, identity=True)
        Cc, C = oracle.conv_channels(d)
        before = pool.copy()
        out, _, fl = orc.in_proj_conv(d, xs, Wm, taps, bias, pool, idx, write_pool=True)
        assert fl == 0
        for b in range(len(idx)):
            for c in range(C):
                if c >= Cc:
                    assert abs(out[b, :, c] - xs[b, :, c]).max() <= 1e-15, (K, T, b, c)
                    continue
                seq = np.concatenate([before[idx[b], :, c], xs[b, :, c]])
                y = float(bias[c]) + np.convolve(seq, taps[c, ::-1].astype(np.float64), mode="valid")
                if silu:
                    y = y * expit(y)
                assert y.shape == (T,)
                assert abs(out[b, :, c] - y).max() <= 1e-13 * max(1.0, abs(y).max()), (K, T, b, c)
                assert np.array_equal(pool[idx[b], :, c], seq[T:]), (K, T, b, c)


def check_conv_state_chain_and_commit(orc):
    """A decode of T rows equals T decodes of one row (outputs and state, exact in fp64); a verify that keeps
    its recovery records followed by the commit of L rows leaves the state that L one-row decodes leave (L = 0:
    unchanged); padded lanes touch nothing; a bad index and a bad accept length set their flag bits."""
    T = 3
    d, xs, Wm, taps, bias, pool0, idx = _conv_case(B=3, T=T, K=4, silu=1, seed=90)
    pool_a = pool0.copy()
    out_a, _, _ = orc.in_proj_conv(d, xs, Wm, taps, bias, pool_a, idx, write_pool=True)
    d1 = dict(d, T=1)
    pools = [pool0.copy()]
    for t in range(T):
        p = pools[-1].copy()
        o1, _, _ = orc.in_proj_conv(d1, np.ascontiguousarray(xs[:, t:t + 1]), Wm, taps, bias, p, idx, write_pool=True)
        assert np.array_equal(o1[:, 0], out_a[:, t]), t
        pools.append(p)
    assert np.array_equal(pools[T], pool_a)
    # verify (read-only) then commit
    pool_v = pool0.copy()
    out_v, rec, _ = orc.in_proj_conv(d, xs, Wm, taps, bias, pool_v, idx, write_pool=False)
    assert np.array_equal(out_v, out_a) and np.array_equal(pool_v, pool0)
    L = np.array([2, 0, 3], np.int32)
    assert orc.conv_commit(d, pool_v, idx, rec, L) == 0
    for b in range(3):
        assert np.array_equal(pool_v[idx[b]], pools[L[b]][idx[b]]), b
    # padding and bad data
    idx2 = idx.copy()
    idx2[1] = -1
    pool_p = pool0.copy()
    canary = np.full(out_a.shape, CANARY)
    out_p, _, fl = orc.in_proj_conv(d, xs, Wm, taps, bias, pool_p, idx2, write_pool=True, out=canary)
    assert fl == 0 and np.all(out_p[1] == CANARY) and np.array_equal(pool_p[idx[1]], pool0[idx[1]])
    assert np.array_equal(out_p[0], out_a[0]) and np.array_equal(pool_p[idx[0]], pool_a[idx[0]])
    idx2[1] = d["num_slots"]
    assert orc.in_proj_conv(d, xs, Wm, taps, bias, pool0.copy(), idx2, write_pool=True)[2] == 1
    pool_c = pool0.copy()
    assert orc.conv_commit(d, pool_c, idx, rec, np.array([1, T + 1, -1], np.int32)) == 2
    assert np.array_equal(pool_c[idx[1]], pool0[idx[1]]) and np.array_equal(pool_c[idx[2]], pool0[idx[2]])


def check_conv_records_rounded(orc):
    """A bf16 or fp32 state stores each pre-convolution value rounded once from the exact product (the rounding
    pinned above), and the convolution reads those stored values; x and W in bf16 or fp32 are read exactly."""
    import oracle
    from gdn_workloads import bf16_bits_to_f32, to_bf16_bits

    for conv in ("bf16", "f32"):
        d, xs, Wm, taps, bias, _, idx = _conv_case(B=2, T=2, K=3, silu=0, conv=conv, seed=95)
        Cc, C = oracle.conv_channels(d)
        xb = to_bf16_bits(xs.astype(np.float32))
        Wb = to_bf16_bits(Wm.astype(np.float32))
        d["x_dtype"] = "bf16"
        pool = np.zeros((d["num_slots"], 2, Cc), np.uint16 if conv == "bf16" else np.float32)
        out, rec, _ = orc.in_proj_conv(d, xb, Wb, taps, bias, pool, idx, write_pool=True)
        exact = np.einsum("ch,bth->btc", bf16_bits_to_f32(Wb).astype(np.float64), bf16_bits_to_f32(xb).astype(np.float64))
        if conv == "bf16":
            want = np.vectorize(orc.round_bf16)(exact[..., :Cc])
            got = bf16_bits_to_f32(rec).astype(np.float64)
            stored = bf16_bits_to_f32(pool[idx]).astype(np.float64)
        else:
            want = exact[..., :Cc].astype(np.float32).astype(np.float64)
            got = rec.astype(np.float64)
            stored = pool[idx].astype(np.float64)
        assert np.array_equal(got, want), conv
        assert np.array_equal(stored[:, 0], want[:, 0]) and np.array_equal(stored[:, 1], want[:, 1]), conv
        # zero state, K = 3: y_t = bias + w2 u_t + w1 u_{t-1}
        y1 = bias + taps[:, 2].astype(np.float64) * want[:, 1] + taps[:, 1].astype(np.float64) * want[:, 0]
        assert np.abs(out[:, 1, :Cc] - y1).max() <= 1e-13, conv
        assert np.abs(out[..., Cc:] - exact[..., Cc:]).max() <= 1e-13, conv


ALL_CHECKS = [check_bf16_rounding, check_scalar_functions, check_gate_closed_form, check_beta_sigmoid,
              check_beta_zero_pure_decay, check_orthonormal_keys_write_v, check_l2norm_eps, check_scale,
              check_head_mapping, check_product_form, check_chained_calls, check_padding_and_bad_data,
              check_commit_replay, check_prefill_product_form, check_prefill_fresh_state,
              check_prefill_matches_verify_and_decode, check_prefill_chained, check_prefill_bad_bounds,
              check_gated_rmsnorm_closed_forms, check_in_proj_is_the_matrix_product, check_conv_is_numpy_convolve,
              check_conv_state_chain_and_commit, check_conv_records_rounded]
