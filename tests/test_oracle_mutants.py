"""The oracle's pins are strong enough: a plausible mistake planted in a copy of the oracle fails at least
one of them.  Every mutant is compiled from a text-substituted copy of ``oracle/gdn_oracle.c`` into a
temporary directory, on the CPU; the committed oracle is never modified.  Each mutant keeps every access
of every pin in bounds (a mutant runs in this process: an out-of-bounds write would corrupt its heap)."""
import os

import pytest

import oracle
import oracle_checks as C
from oracle import build as obuild

# (name, text in gdn_oracle.c, replacement)
MUTANTS = [
    ("gate_sign", "return exp(-exp(A_log) * orc_softplus(a + dt_bias));",
     "return exp(exp(A_log) * orc_softplus(a + dt_bias));"),
    ("dt_bias_sign", "return exp(-exp(A_log) * orc_softplus(a + dt_bias));",
     "return exp(-exp(A_log) * orc_softplus(a - dt_bias));"),
    ("gate_no_exp_of_A_log", "return exp(-exp(A_log) * orc_softplus(a + dt_bias));",
     "return exp(-A_log * orc_softplus(a + dt_bias));"),
    ("gate_softplus_dropped", "return exp(-exp(A_log) * orc_softplus(a + dt_bias));",
     "return exp(-exp(A_log) * (a + dt_bias));"),
    ("softplus_positive_branch", "return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));",
     "return x > 0.0 ? x : log1p(exp(x));"),
    ("sigmoid_sign", "double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }",
     "double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(x)); }"),
    ("eps_outside_root", "const double qn = sqrt(qq + d->l2_eps), kn = sqrt(kk + d->l2_eps);",
     "const double qn = sqrt(qq) + d->l2_eps, kn = sqrt(kk) + d->l2_eps;"),
    ("k_not_normalised", "kh[j] = load(k, d->qkv_dtype, qk_off + j) / kn;",
     "kh[j] = load(k, d->qkv_dtype, qk_off + j);"),
    ("decay_dropped", "for (int i = 0; i < DV * DK; ++i) S[i] *= g;", ""),
    ("u_uses_query", "for (int j = 0; j < DK; ++j) s += S[i * DK + j] * kh[j];",
     "for (int j = 0; j < DK; ++j) s += S[i * DK + j] * qh[j];"),
    ("beta_dropped", "const double delta = beta * (load(v, d->qkv_dtype, v_off + i) - u[i]);",
     "const double delta = (load(v, d->qkv_dtype, v_off + i) - u[i]);"),
    ("delta_sign", "const double delta = beta * (load(v, d->qkv_dtype, v_off + i) - u[i]);",
     "const double delta = beta * (load(v, d->qkv_dtype, v_off + i) + u[i]);"),
    ("v_index", "load(v, d->qkv_dtype, v_off + i)", "load(v, d->qkv_dtype, v_off)"),
    ("head_mapping_modulo", "const int hk = h / r;", "const int hk = h % HK;"),
    ("output_skips_scale", "o[v_off + i] = d->scale * s;", "o[v_off + i] = s;"),
    ("cache_token_index", "const int64_t c_off = ((((int64_t)b * T + t) * HV) + h) * DV * DK;",
     "const int64_t c_off = ((((int64_t)b * T + 0) * HV) + h) * DV * DK;"),
    ("bf16_truncates", "double y = ldexp(nearbyint(ldexp(x, -q)), q);",
     "double y = ldexp(trunc(ldexp(x, -q)), q);"),
    ("bf16_keeps_9_bits", "int q = e - 8;", "int q = e - 9;"),
    ("commit_first_token", "(((int64_t)b * d->T) + (L - 1)) * per_lane", "(((int64_t)b * d->T) + 0) * per_lane"),
    ("padding_not_skipped", "if (slot == -1) return -1;", "if (slot == -1) return 0;"),
    ("accept_len_unchecked", "if (L < 0 || L > d->T) {", "if (0) {"),
    ("replay_ignores_accept_len", "int n_tok = steps ? steps[b] : T;", "int n_tok = T;"),
    ("replay_off_by_one", "int n_tok = steps ? steps[b] : T;", "int n_tok = steps ? steps[b] - (steps[b] > 1) : T;"),
    ("prefill_fresh_reads_pool", "const int fresh = has_init && !has_init[b];", "const int fresh = 0;"),
    ("prefill_fresh_inverted", "const int fresh = has_init && !has_init[b];",
     "const int fresh = has_init && has_init[b];"),
    ("prefill_token_base", "tok0 = seq[b];", "tok0 = seq[b] > 0 ? seq[b] - 1 : 0;"),
    ("prefill_length_one_short", "n_tok = seq[b + 1] - seq[b];", "n_tok = seq[b + 1] - seq[b] - (seq[b + 1] > seq[b]);"),
    ("prefill_bad_bounds_flag", "flags |= 8;", "flags |= 2;"),
    ("norm_sum_not_mean", "ms /= DV;", ""),
    ("norm_eps_outside_root", "const double inv_rms = 1.0 / sqrt(ms + eps);",
     "const double inv_rms = 1.0 / (sqrt(ms) + eps);"),
    ("norm_gate_sigmoid_only", "const double silu = zi * orc_sigmoid(zi);", "const double silu = orc_sigmoid(zi);"),
    ("norm_gate_sign", "const double silu = zi * orc_sigmoid(zi);", "const double silu = zi * orc_sigmoid(-zi);"),
    ("norm_weight_index", "* (double)w[i] * silu;", "* (double)w[0] * silu;"),
    ("norm_gate_row", "const double zi = load(z, z_dtype, r * DV + i);", "const double zi = load(z, z_dtype, i);"),
    ("in_proj_W_transposed", "load(W, d->x_dtype, c * H + h)", "load(W, d->x_dtype, h * C + c)"),
    ("in_proj_row_index", "load(x, d->x_dtype, ((int64_t)b * T + t) * H + h)", "load(x, d->x_dtype, ((int64_t)b * T) * H + h)"),
    ("conv_taps_reversed", "y += (double)conv_w[c * K + j] * seq[t + j];",
     "y += (double)conv_w[c * K + (K - 1 - j)] * seq[t + j];"),
    ("conv_bias_dropped", "double y = conv_b ? (double)conv_b[c] : 0.0;", "double y = 0.0;"),
    ("conv_silu_sigmoid_only", "if (d->silu) y = y * orc_sigmoid(y);", "if (d->silu) y = orc_sigmoid(y);"),
    ("conv_records_unrounded", "seq[K - 1 + t] = round_to(d->conv_dtype, p);", "seq[K - 1 + t] = p;"),
    ("conv_state_from_lane", "seq[j] = load(conv_pool, d->conv_dtype, ((int64_t)slot * (K - 1) + j) * Cc + c);",
     "seq[j] = load(conv_pool, d->conv_dtype, ((int64_t)b * (K - 1) + j) * Cc + c);"),
    ("conv_write_back_one_early", "((int64_t)slot * (K - 1) + j) * Cc + c, seq[T + j]);",
     "((int64_t)slot * (K - 1) + j) * Cc + c, seq[T + j - 1]);"),
    ("conv_commit_one_early", "((int64_t)slot * (K - 1) + j) * Cc + c, seq[L + j]);",
     "((int64_t)slot * (K - 1) + j) * Cc + c, seq[L + j - 1]);"),
    ("conv_commit_ignores_accept_len", "((int64_t)slot * (K - 1) + j) * Cc + c, seq[L + j]);",
     "((int64_t)slot * (K - 1) + j) * Cc + c, seq[T + j]);"),
    ("conv_padding_not_skipped", "    const int32_t slot = idx[b];\n    if (slot == -1) return -1;\n    if (slot < 0 || slot >= d->num_slots) {",
     "    const int32_t slot = idx[b] == -1 ? 0 : idx[b];\n    if (slot < 0 || slot >= d->num_slots) {"),
    ("norm_output_unnormalised", "y[r * DV + i] = load(o, o_dtype, r * DV + i) * inv_rms * (double)w[i] * silu;",
     "y[r * DV + i] = load(o, o_dtype, r * DV + i) * (double)w[i] * silu;"),
]


@pytest.fixture(scope="module")
def source():
    with open(obuild.SOURCE) as f:
        return f.read()


def test_mutant_targets_present(source):
    for name, old, _ in MUTANTS:
        assert source.count(old) >= 1, name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    mutated = source.replace(old, new)
    assert mutated != source
    src = tmp_path / "gdn_oracle_mutant.c"
    src.write_text(mutated)
    lib = obuild.build(str(src), str(tmp_path / "libmutant.so"), extra=["-w"])
    orc = oracle.Oracle(lib)
    failures = []
    for check in C.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError, FloatingPointError) as e:  # a pin caught it
            failures.append(check.__name__)
    assert failures, f"mutant {name} passed every pin"
    os.remove(lib)
