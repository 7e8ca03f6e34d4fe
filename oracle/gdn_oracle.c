/*
 * gdn_oracle.c -- plain, slow, obviously-correct CPU reference of the Gated DeltaNet (GDN) recurrent
 * state update used for decode and for multi-token-prediction (MTP) speculative verify.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * arm may call this.  It shares no code, header or helper with the CUDA library.
 *
 * What it computes (the gated delta rule behind FlashInfer's gated_delta_rule_mtp, named in sglang
 * PR #23273 "[GDN] Enable FlashInfer MTP verify on SM100+ (Blackwell)", Summary; the pages never write the
 * recurrence out, so it is restated here):
 *
 *   for every lane b whose pool index slot = idx[b] is >= 0, and every value head h
 *   (key head hk = h / (HV / HK), contiguous groups):
 *     S = pool[slot, h]                                  (DV x DK, read as the exact stored value)
 *     for t = 0 .. T-1:
 *       qh = q[b,t,hk] / sqrt(sum(q^2) + eps)            (L2 normalisation, eps inside the root)
 *       kh = k[b,t,hk] / sqrt(sum(k^2) + eps)
 *       g    = exp(-exp(A_log[h]) * softplus(a[b,t,h] + dt_bias[h]))
 *       beta = 1 / (1 + exp(-b[b,t,h]))
 *       S = g * S
 *       u = S kh
 *       S = S + beta * (v[b,t,h] - u) kh^T
 *       o[b,t,h] = scale * S qh
 *       verify with caching: cache[b,t,h] = R(S)
 *     decode: pool[slot, h] = R(S)
 *   commit: pool[idx[b], h] = cache[b, L_b - 1, h] for lanes with L_b >= 1.
 *   replay commit: the first L_b tokens again from pool[idx[b], h], then pool[idx[b], h] = R(S): the
 *     same value as the commit above, without caching every intermediate state.
 *
 *   prefill: B variable-length sequences packed along one token axis of length N (= dims T): sequence b
 *     runs tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 from S = pool[idx[b], h] if has_initial_state[b] is
 *     non-zero, else from S = 0 (the pool slot is then not read at all: fresh-state zeroing), writes o at
 *     those token positions and pool[idx[b], h] = R(S) after its last token.  The chunked gated delta
 *     rule with a bf16 state pool and an initial-state mask of TensorRT-LLM PR #20937 (GB300 Qwen3.8-Flash-
 *     Next NVFP4), Per-File QA Perspective, Source files and Test-code files (flashinfer_chunk_gated_delta_
 *     rule: "fresh-state zeroing", bf16 pools); the chunking there is an evaluation order of this same
 *     recurrence, so the definition is the token loop.
 *   gated RMSNorm of the outputs (the "decode rows gated norm" of the same page and section), per row r of
 *     DV outputs:  y[r, i] = o[r, i] / sqrt(mean_i(o[r, i]^2) + eps) * w[i] * silu(z[r, i]),
 *     silu(x) = x * sigmoid(x).  The page names the fusion, not its formula: this is the plain reading
 *     (RMS over the value dimension of one head, one weight vector of length DV shared by all heads, the
 *     gate applied after the norm).
 *
 * Padded lanes (index -1) are skipped: the page's padding index guard (sglang PR #23273, Requirements,
 * FlashInfer #2810).  bf16 state with intermediate caching beyond T > 4: same page, Requirements
 * (FlashInfer #2679).  A_log is fp32: same page, Summary (A_log.detach().float()).
 *
 * Arithmetic is fp64.  R rounds the fp64 running state to the storage type only where a state is stored
 * (each cache write, the decode write-back): round-to-nearest-even, directly from fp64 (no double
 * rounding).  The running state of one call is never rounded between tokens.
 *
 * Out-of-range data (index < -1 or >= num_slots, accept length outside 0..T, a prefill sequence whose
 * bounds are negative, decreasing or beyond N) skips the lane and sets a bit in the returned flag word:
 * bit 0 = index, bit 1 = accept length, bit 3 = sequence bounds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

typedef struct {
    int32_t B, T, HK, HV, DK, DV, num_slots;
    int32_t qkv_dtype;   /* q, k, v, a, b storage type */
    int32_t state_dtype; /* pool storage type */
    int32_t cache_dtype; /* intermediate cache storage type */
    double scale;
    double l2_eps;
} orc_dims;

/* ---- storage types --------------------------------------------------------------------------- */

static double bf16_bits_to_double(uint16_t h) {
    uint32_t w = (uint32_t)h << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Nearest bfloat16 value to x, ties to even, overflow to infinity; returned as a double. */
double orc_round_bf16(double x) {
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    int e;
    frexp(x, &e);       /* |x| in [2^(e-1), 2^e) */
    int q = e - 8;      /* bf16 keeps 8 significant bits: the last one weighs 2^(e-8) */
    if (q < -133) q = -133; /* below the normal range the step is that of the subnormals, 2^-133 */
    double y = ldexp(nearbyint(ldexp(x, -q)), q);
    if (fabs(y) >= 0x1p128) y = copysign(INFINITY, x);
    return y;
}

static uint16_t double_to_bf16_bits(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    float f = (float)orc_round_bf16(x); /* exact: the rounded value is a bf16 value */
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(w >> 16);
}

static double load(const void* base, int dtype, int64_t i) {
    switch (dtype) {
    case ORC_F32: return (double)((const float*)base)[i];
    case ORC_BF16: return bf16_bits_to_double(((const uint16_t*)base)[i]);
    case ORC_F64: return ((const double*)base)[i];
    }
    return NAN;
}

static void store(void* base, int dtype, int64_t i, double x) {
    switch (dtype) {
    case ORC_F32: ((float*)base)[i] = (float)x; break; /* C conversion: nearest, ties to even */
    case ORC_BF16: ((uint16_t*)base)[i] = double_to_bf16_bits(x); break;
    case ORC_F64: ((double*)base)[i] = x; break;
    }
}

static size_t dtype_size(int dtype) { return dtype == ORC_F32 ? 4 : dtype == ORC_BF16 ? 2 : 8; }

/* ---- scalar functions ------------------------------------------------------------------------- */

/* softplus(x) = log(1 + e^x); for x > 0 written as x + log(1 + e^-x), the same value without overflow */
double orc_softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

double orc_gate(double A_log, double a, double dt_bias) {
    return exp(-exp(A_log) * orc_softplus(a + dt_bias));
}

/* ---- the recurrence ----------------------------------------------------------------------------- */

static int lane_slot(const orc_dims* d, const int32_t* idx, int b, int* flags) {
    int32_t slot = idx[b];
    if (slot == -1) return -1;
    if (slot < -1 || slot >= d->num_slots) {
        *flags |= 1;
        return -1;
    }
    return slot;
}

/* Runs the tokens of every active lane: all T, or steps[b] of them if steps != NULL (a count outside 0..T
 * sets flag bit 1 and skips the lane), or, if seq != NULL (prefill), tokens seq[b] .. seq[b+1]-1 of the
 * token axis (bounds outside 0..T set flag bit 3 and skip the lane).  A lane with has_init != NULL and
 * has_init[b] == 0 starts from the zero state.  If o != NULL, stores the outputs.  If cache != NULL,
 * stores R(S) after every token (verify).  If write_back, stores R(S) of the last token run into the
 * lane's pool slot (decode; replay commit; prefill). */
static int run(const orc_dims* d, const void* q, const void* k, const void* v, const void* a,
               const void* bb, const float* A_log, const float* dt_bias, void* pool, const int32_t* idx,
               double* o, void* cache, int write_back, const int32_t* steps, const int32_t* seq,
               const int32_t* has_init) {
    const int B = d->B, T = d->T, HK = d->HK, HV = d->HV, DK = d->DK, DV = d->DV;
    const int r = HV / HK;
    int flags = 0;
    double* S = (double*)malloc(sizeof(double) * (size_t)DV * DK);
    double* qh = (double*)malloc(sizeof(double) * DK);
    double* kh = (double*)malloc(sizeof(double) * DK);
    double* u = (double*)malloc(sizeof(double) * DV);
    if (!S || !qh || !kh || !u) {
        free(S); free(qh); free(kh); free(u);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        int slot = lane_slot(d, idx, b, &flags);
        if (slot < 0) continue;
        /* the lane's tokens are positions tok0 .. tok0 + n_tok - 1 of the token axis of q, k, v, a, b, o */
        int64_t tok0 = (int64_t)b * T;
        int n_tok = steps ? steps[b] : T;
        if (seq) {
            if (seq[b] < 0 || seq[b + 1] < seq[b] || seq[b + 1] > T) {
                flags |= 8;
                continue;
            }
            tok0 = seq[b];
            n_tok = seq[b + 1] - seq[b];
        }
        if (n_tok < 0 || n_tok > T) {
            flags |= 2;
            continue;
        }
        if (n_tok == 0) continue;
        const int fresh = has_init && !has_init[b];
        for (int h = 0; h < HV; ++h) {
            const int hk = h / r;
            const int64_t state_off = ((int64_t)slot * HV + h) * DV * DK;
            for (int i = 0; i < DV; ++i)
                for (int j = 0; j < DK; ++j)
                    S[i * DK + j] = fresh ? 0.0 : load(pool, d->state_dtype, state_off + i * DK + j);

            for (int t = 0; t < n_tok; ++t) {
                const int64_t qk_off = ((tok0 + t) * HK + hk) * DK;
                const int64_t ab_off = (tok0 + t) * HV + h;
                const int64_t v_off = ((tok0 + t) * HV + h) * DV;

                double qq = 0.0, kk = 0.0;
                for (int j = 0; j < DK; ++j) {
                    double qj = load(q, d->qkv_dtype, qk_off + j), kj = load(k, d->qkv_dtype, qk_off + j);
                    qq += qj * qj;
                    kk += kj * kj;
                }
                const double qn = sqrt(qq + d->l2_eps), kn = sqrt(kk + d->l2_eps);
                for (int j = 0; j < DK; ++j) {
                    qh[j] = load(q, d->qkv_dtype, qk_off + j) / qn;
                    kh[j] = load(k, d->qkv_dtype, qk_off + j) / kn;
                }
                const double g = orc_gate(A_log[h], load(a, d->qkv_dtype, ab_off), dt_bias[h]);
                const double beta = orc_sigmoid(load(bb, d->qkv_dtype, ab_off));

                for (int i = 0; i < DV * DK; ++i) S[i] *= g;
                for (int i = 0; i < DV; ++i) {
                    double s = 0.0;
                    for (int j = 0; j < DK; ++j) s += S[i * DK + j] * kh[j];
                    u[i] = s;
                }
                for (int i = 0; i < DV; ++i) {
                    const double delta = beta * (load(v, d->qkv_dtype, v_off + i) - u[i]);
                    for (int j = 0; j < DK; ++j) S[i * DK + j] += delta * kh[j];
                }
                for (int i = 0; o && i < DV; ++i) {
                    double s = 0.0;
                    for (int j = 0; j < DK; ++j) s += S[i * DK + j] * qh[j];
                    o[v_off + i] = d->scale * s;
                }
                if (cache) {
                    const int64_t c_off = ((((int64_t)b * T + t) * HV) + h) * DV * DK;
                    for (int i = 0; i < DV * DK; ++i) store(cache, d->cache_dtype, c_off + i, S[i]);
                }
            }
            if (write_back)
                for (int i = 0; i < DV * DK; ++i) store(pool, d->state_dtype, state_off + i, S[i]);
        }
    }
    free(S); free(qh); free(kh); free(u);
    return flags;
}

static int dims_ok(const orc_dims* d) {
    return d->B >= 0 && d->T >= 1 && d->HK >= 1 && d->HV >= 1 && d->HV % d->HK == 0 && d->DK >= 1 &&
           d->DV >= 1 && d->num_slots >= 1;
}

/* T tokens from pool[idx[b]] (read only); o in fp64; cache (nullable) in cache_dtype. */
int orc_verify(const orc_dims* d, const void* q, const void* k, const void* v, const void* a, const void* b,
               const float* A_log, const float* dt_bias, const void* pool, const int32_t* idx, double* o,
               void* cache) {
    if (!dims_ok(d)) return -2;
    return run(d, q, k, v, a, b, A_log, dt_bias, (void*)pool, idx, o, cache, 0, NULL, NULL, NULL);
}

/* T tokens from pool[idx[b]], final state written back into the same slot. */
int orc_decode(const orc_dims* d, const void* q, const void* k, const void* v, const void* a, const void* b,
               const float* A_log, const float* dt_bias, void* pool, const int32_t* idx, double* o) {
    if (!dims_ok(d)) return -2;
    return run(d, q, k, v, a, b, A_log, dt_bias, pool, idx, o, NULL, 1, NULL, NULL, NULL);
}

/* Replay commit: the first accept_len[b] tokens of every active lane from pool[idx[b]], the final state
 * written back into that slot (no outputs).  Equals orc_commit after orc_verify with caching. */
int orc_commit_replay(const orc_dims* d, const void* q, const void* k, const void* v, const void* a,
                      const void* b, const float* A_log, const float* dt_bias, void* pool, const int32_t* idx,
                      const int32_t* accept_len) {
    if (!dims_ok(d)) return -2;
    return run(d, q, k, v, a, b, A_log, dt_bias, pool, idx, NULL, NULL, 1, accept_len, NULL, NULL);
}

/* Prefill: d->B sequences over a token axis of d->T tokens (q, k [T, HK, DK]; v [T, HV, DV]; a, b [T, HV];
 * o [T, HV, DV]); has_init (nullable: every sequence has one) selects the pool state or zero as the start;
 * the final state goes into pool[idx[b]].  Positions outside every sequence, and those of skipped lanes,
 * keep their o. */
int orc_prefill(const orc_dims* d, const int32_t* cu_seqlens, const void* q, const void* k, const void* v,
                const void* a, const void* b, const float* A_log, const float* dt_bias, void* pool,
                const int32_t* idx, const int32_t* has_init, double* o) {
    if (!dims_ok(d)) return -2;
    return run(d, q, k, v, a, b, A_log, dt_bias, pool, idx, o, NULL, 1, NULL, cu_seqlens, has_init);
}

/* Gated RMSNorm of `rows` rows of DV values: o and z in their storage types, w fp32 [DV], y fp64. */
int orc_gated_rmsnorm(int64_t rows, int32_t DV, const void* o, int32_t o_dtype, const void* z, int32_t z_dtype,
                      const float* w, double eps, double* y) {
    if (rows < 0 || DV < 1 || eps < 0.0) return -2;
    for (int64_t r = 0; r < rows; ++r) {
        double ms = 0.0;
        for (int i = 0; i < DV; ++i) {
            const double x = load(o, o_dtype, r * DV + i);
            ms += x * x;
        }
        ms /= DV;
        const double inv_rms = 1.0 / sqrt(ms + eps);
        for (int i = 0; i < DV; ++i) {
            const double zi = load(z, z_dtype, r * DV + i);
            const double silu = zi * orc_sigmoid(zi);
            y[r * DV + i] = load(o, o_dtype, r * DV + i) * inv_rms * (double)w[i] * silu;
        }
    }
    return 0;
}

/* pool[idx[b], :] = cache[b, L_b - 1, :] (all heads), bit for bit, for active lanes with L_b >= 1. */
int orc_commit(const orc_dims* d, void* pool, const int32_t* idx, const void* cache, const int32_t* accept_len) {
    if (!dims_ok(d)) return -2;
    if (d->cache_dtype != d->state_dtype) return -3;
    int flags = 0;
    const size_t es = dtype_size(d->state_dtype);
    const int64_t per_lane = (int64_t)d->HV * d->DV * d->DK;
    for (int b = 0; b < d->B; ++b) {
        int slot = lane_slot(d, idx, b, &flags);
        if (slot < 0) continue;
        const int L = accept_len[b];
        if (L < 0 || L > d->T) {
            flags |= 2;
            continue;
        }
        if (L == 0) continue;
        const char* src = (const char*)cache + (((int64_t)b * d->T) + (L - 1)) * per_lane * (int64_t)es;
        char* dst = (char*)pool + (int64_t)slot * per_lane * (int64_t)es;
        memcpy(dst, src, (size_t)(per_lane * (int64_t)es));
    }
    return flags;
}

/* ---- the in_proj projection with its causal conv1d epilogue ------------------------------------------------
 *
 * The GDN input projection of the decode and verify rows with the short causal convolution fused after it:
 * TensorRT-LLM PR #20937 (GB300 Qwen3.8-Flash-Next NVFP4), What changes, Decode at small batch ("the in_proj
 * GEMV with a fused conv1d epilogue, for 2..16 verify rows and up to 8 decode rows"); the convolution state is
 * committed with the accepted prefix (issue "Proposal: native BF16 MTP speculative decoding for dense
 * Qwen3.8-27B", What: the compact GDN recovery records and their commit, with the convolution's).  The pages give
 * no formula; the plain reading written out here:
 *
 *   rows: lane b owns rows b*T .. b*T+T-1 of x [B*T, H]; W [C, H] with its C output channels in the order
 *     q (HK*DK) | k (HK*DK) | v (HV*DV) | z (HV*DV) | b (HV) | a (HV); the first Cc = 2*HK*DK + HV*DV channels
 *     (q, k, v) go through the convolution.
 *   p[t, c]  = sum_h W[c, h] * x[b*T + t, h]
 *   u[t, c]  = R_conv(p[t, c])                  (c < Cc: the pre-convolution value as the state stores it)
 *   seq      = pool[slot, 0 .. K-2, c] (oldest first), then u[0 .. T-1, c]
 *   y[t, c]  = bias[c] + sum_{j < K} w[c, j] * seq[t + j, c]    (tap K-1 weighs the current row)
 *   y        = y * sigmoid(y) when silu is set
 *   out[b, t, c] = y[t, c] for c < Cc, p[t, c] otherwise (fp64; the caller rounds to its output type)
 *   u_rec[b, t, c] = u[t, c]  (the verify rows' recovery records, if asked for)
 *   write_pool (decode): pool[slot, j, c] = seq[T + j, c] for j < K-1 (the last K-1 entries)
 *   conv commit of L accepted rows: pool[slot, j, c] = seq[L + j, c] with seq built from u_rec (bit copies);
 *     L = 0 leaves the slot, L outside 0..T sets flag bit 1.
 * Padded lanes (index -1) are skipped entirely; other out-of-range indices set flag bit 0.
 */
typedef struct {
    int32_t B, T, H;        /* lanes, rows per lane, hidden size */
    int32_t HK, HV, DK, DV; /* head layout of the outputs */
    int32_t K;              /* convolution taps */
    int32_t num_slots;
    int32_t x_dtype;        /* storage type of x and W */
    int32_t conv_dtype;     /* storage type of the convolution-state pool and of the recovery records */
    int32_t silu;           /* 1: SiLU after the convolution */
} orc_conv_dims;

static double round_to(int dtype, double x) {
    switch (dtype) {
    case ORC_F32: return (double)(float)x;
    case ORC_BF16: return orc_round_bf16(x);
    }
    return x;
}

static int conv_dims_ok(const orc_conv_dims* d) {
    return d->B >= 0 && d->T >= 1 && d->H >= 1 && d->HK >= 1 && d->HV >= 1 && d->DK >= 1 && d->DV >= 1 &&
           d->K >= 1 && d->K <= 8 && d->num_slots >= 0;
}

static int conv_lane_slot(const orc_conv_dims* d, const int32_t* idx, int b, int* flags) {
    const int32_t slot = idx[b];
    if (slot == -1) return -1;
    if (slot < 0 || slot >= d->num_slots) {
        *flags |= 1;
        return -1;
    }
    return slot;
}

int orc_in_proj_conv(const orc_conv_dims* d, const void* x, const void* W, const float* conv_w, const float* conv_b,
                     void* conv_pool, const int32_t* idx, int32_t write_pool, double* out, void* u_rec) {
    if (!conv_dims_ok(d)) return -2;
    const int T = d->T, H = d->H, K = d->K;
    const int64_t Cc = 2 * (int64_t)d->HK * d->DK + (int64_t)d->HV * d->DV;
    const int64_t C = Cc + (int64_t)d->HV * d->DV + 2 * (int64_t)d->HV;
    int flags = 0;
    double* seq = (double*)malloc(sizeof(double) * (size_t)(K - 1 + T));
    if (seq == NULL) return -4;
    for (int b = 0; b < d->B; ++b) {
        const int slot = conv_lane_slot(d, idx, b, &flags);
        if (slot < 0) continue;
        for (int64_t c = 0; c < C; ++c) {
            for (int t = 0; t < T; ++t) {
                double p = 0.0;
                for (int h = 0; h < H; ++h)
                    p += load(W, d->x_dtype, c * H + h) * load(x, d->x_dtype, ((int64_t)b * T + t) * H + h);
                if (c < Cc) {
                    seq[K - 1 + t] = round_to(d->conv_dtype, p);
                } else {
                    out[((int64_t)b * T + t) * C + c] = p;
                }
            }
            if (c >= Cc) continue;
            for (int j = 0; j < K - 1; ++j)
                seq[j] = load(conv_pool, d->conv_dtype, ((int64_t)slot * (K - 1) + j) * Cc + c);
            for (int t = 0; t < T; ++t) {
                double y = conv_b ? (double)conv_b[c] : 0.0;
                for (int j = 0; j < K; ++j) y += (double)conv_w[c * K + j] * seq[t + j];
                if (d->silu) y = y * orc_sigmoid(y);
                out[((int64_t)b * T + t) * C + c] = y;
                if (u_rec) store(u_rec, d->conv_dtype, ((int64_t)b * T + t) * Cc + c, seq[K - 1 + t]);
            }
            if (write_pool)
                for (int j = 0; j < K - 1; ++j)
                    store(conv_pool, d->conv_dtype, ((int64_t)slot * (K - 1) + j) * Cc + c, seq[T + j]);
        }
    }
    free(seq);
    return flags;
}

int orc_conv_commit(const orc_conv_dims* d, void* conv_pool, const int32_t* idx, const void* u_rec,
                    const int32_t* accept_len) {
    if (!conv_dims_ok(d)) return -2;
    const int T = d->T, K = d->K;
    const int64_t Cc = 2 * (int64_t)d->HK * d->DK + (int64_t)d->HV * d->DV;
    int flags = 0;
    double* seq = (double*)malloc(sizeof(double) * (size_t)(K - 1 + T));
    if (seq == NULL) return -4;
    for (int b = 0; b < d->B; ++b) {
        const int slot = conv_lane_slot(d, idx, b, &flags);
        if (slot < 0) continue;
        const int L = accept_len[b];
        if (L < 0 || L > T) {
            flags |= 2;
            continue;
        }
        if (L == 0) continue;
        for (int64_t c = 0; c < Cc; ++c) {
            for (int j = 0; j < K - 1; ++j)
                seq[j] = load(conv_pool, d->conv_dtype, ((int64_t)slot * (K - 1) + j) * Cc + c);
            for (int t = 0; t < T; ++t) seq[K - 1 + t] = load(u_rec, d->conv_dtype, ((int64_t)b * T + t) * Cc + c);
            for (int j = 0; j < K - 1; ++j)
                store(conv_pool, d->conv_dtype, ((int64_t)slot * (K - 1) + j) * Cc + c, seq[L + j]);
        }
    }
    free(seq);
    return flags;
}
