/*
 * gdn.h -- C ABI of libgdn.so: the Gated DeltaNet (GDN) recurrent state update for decode and for
 * multi-token-prediction (MTP) speculative verify, on one GB300 (sm_103a).
 *
 * The operation (the gated delta rule behind FlashInfer's gated_delta_rule_mtp, which sglang PR #23273
 * "[GDN] Enable FlashInfer MTP verify on SM100+ (Blackwell)" calls through its pool API, Summary):
 * for every request lane b whose pool index slot = state_indices[b] is not -1, and every value head h
 * (key/query head hk = h / (HV / HK): each group of HV/HK consecutive value heads shares one key head),
 *
 *     S = state_pool[slot, h]                                   (DV x DK, computed in fp32)
 *     for t in 0 .. T-1:
 *         qh = q[b,t,hk] / sqrt(|q[b,t,hk]|^2 + l2_eps)         (L2 normalisation)
 *         kh = k[b,t,hk] / sqrt(|k[b,t,hk]|^2 + l2_eps)
 *         g    = exp(-exp(A_log[h]) * softplus(a[b,t,h] + dt_bias[h]))
 *         beta = sigmoid(b[b,t,h])
 *         S = g * S
 *         S = S + beta * (v[b,t,h] - S kh) kh^T                 (delta rule)
 *         o[b,t,h] = scale * S qh
 *
 * Layouts: row-major, last index contiguous, no strides.
 *     q, k                    [B, T, HK, DK]          qkv_dtype
 *     v                       [B, T, HV, DV]          qkv_dtype
 *     a, b                    [B, T, HV]              qkv_dtype
 *     A_log, dt_bias          [HV]                    fp32 (A_log is fp32: same page, Summary)
 *     state_pool              [num_slots, HV, DV, DK] state_dtype (fp32, or bf16 as with
 *                                                     --mamba-ssm-dtype bfloat16, same page, Throughput)
 *     state_indices           [B]                     int32; -1 = padded lane
 *     o                       [B, T, HV, DV]          out_dtype
 *     intermediate_states     [B, T, HV, DV, DK]      state_dtype
 *     accept_len              [B]                     int32
 *
 * Common rules.
 *   - Every pointer is DEVICE memory owned by the caller, on the device that is current when the call is made
 *     (the one `stream` belongs to).  The library allocates nothing, keeps no state between calls besides
 *     launch-configuration caches (atomic, one entry per device, filled on first use), never synchronises,
 *     and enqueues its work asynchronously on `stream` (0 = legacy default stream).  Calls are thread-safe.
 *     A call with B == 0 (prefill: or no tokens; gated norm: rows == 0) enqueues nothing and returns GDN_OK.
 *   - Alignment: q, k, state_pool and intermediate_states start on 16 bytes; the other arrays on their
 *     element size.  Outputs must not overlap inputs (decode updates state_pool in place by design).
 *   - Errors the host can see are returned as a status before anything is enqueued.  Errors that depend on
 *     device data are defined, never a fault: a lane whose index is < -1 or >= num_slots, (commit) whose
 *     accept length is outside 0..T, or (prefill) whose token bounds are negative, decreasing or beyond the
 *     token count, is skipped and a bit is OR-ed into *err_word (if err_word is not NULL):
 *     GDN_ERRBIT_INDEX, GDN_ERRBIT_ACCEPT_LEN, GDN_ERRBIT_SEQLEN.  No kernel waits on another CTA or on a
 *     flag; the only waits are on the CTA's own bulk copies of state into shared memory, and they are
 *     bounded: one that runs out sets GDN_ERRBIT_TIMEOUT and that part of the state is left unprocessed.
 *     The caller zeroes *err_word and reads it when it wants.
 *   - Padded lanes (index -1, the padding index guard of FlashInfer #2810, same page, Requirements) are
 *     skipped: their o, intermediate states and pool slots are left untouched, bit for bit.
 *   - Distinct active lanes must use distinct slots in gdn_decode and gdn_commit (they write the pool);
 *     gdn_mtp_verify only reads the pool, so lanes may share a slot there.
 *   - GDN_ERR_CUDA: the launch failed; gdn_last_cuda_error() returns the cudaError_t of this thread's last
 *     failed launch.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stdint.h>

/* The library exports these functions and nothing else (it is built with hidden default visibility). */
#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that C callers need no CUDA header. */
typedef struct CUstream_st* gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL */
    GDN_ERR_SHAPE = 2,       /* a size is out of range or inconsistent (HV % HK, T range, ...) */
    GDN_ERR_DTYPE = 3,       /* a dtype code is not a gdn_dtype */
    GDN_ERR_ALIGN = 4,       /* a pointer is misaligned */
    GDN_ERR_UNSUPPORTED = 5, /* a valid but unsupported configuration (DK not in {16,32,64,128,256}) */
    GDN_ERR_CUDA = 6,        /* the kernel launch failed */
    GDN_ERR_VALUE = 7        /* a scalar is not finite, or l2_eps < 0 */
} gdn_status;

typedef enum gdn_dtype { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

enum { GDN_ERRBIT_INDEX = 1, GDN_ERRBIT_ACCEPT_LEN = 2, GDN_ERRBIT_TIMEOUT = 4, GDN_ERRBIT_SEQLEN = 8 };

enum { GDN_MAX_T = 16 }; /* tokens per call: decode (T >= 1), verify up to 16 (the page's MTP beyond T > 4) */

typedef struct gdn_dims {
    int32_t B;           /* request lanes, 0 .. 65535 */
    int32_t T;           /* tokens per lane, 1 .. GDN_MAX_T */
    int32_t HK;          /* query/key heads, >= 1 */
    int32_t HV;          /* value heads, multiple of HK, <= 65535 */
    int32_t DK;          /* key dimension: 16, 32, 64, 128 or 256 */
    int32_t DV;          /* value dimension (state rows), >= 1 */
    int32_t num_slots;   /* pool slots, >= 1 */
    int32_t qkv_dtype;   /* gdn_dtype of q, k, v, a, b */
    int32_t state_dtype; /* gdn_dtype of state_pool and intermediate_states */
    int32_t out_dtype;   /* gdn_dtype of o */
    float scale;         /* multiplies o (1.0 for o = S q) */
    float l2_eps;        /* added to |x|^2 inside the square root of the L2 normalisation (1e-6) */
} gdn_dims;

/*
 * gdn_decode -- T tokens (normally T = 1) from state_pool[state_indices[b]]; the final state is written
 * back into the same slot, rounded to state_dtype (round to nearest even for bf16).  The running state
 * stays fp32 between the tokens of one call.  Defines the SM100+ decode path of sglang PR #23273,
 * Summary, with the padding index guard of its Requirements.
 */
GDN_API gdn_status gdn_decode(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                      const void* b, const float* A_log, const float* dt_bias, void* state_pool,
                      const int32_t* state_indices, void* o, int32_t* err_word, gdn_stream_t stream);

/*
 * gdn_mtp_verify -- T draft tokens from state_pool[state_indices[b]] (read only: the pool is never
 * written).  If intermediate_states is not NULL, the state after token t is stored, rounded to
 * state_dtype, in intermediate_states[b, t].  Without intermediate_states, bf16 state, T <= 8 and DK >= 64,
 * the outputs come from the chunked form of the same recurrence (S_0 [k q] on the tensor cores, k and q split
 * into bf16 hi + lo parts, about 16 significant bits), within fp32-level error of the token-by-token
 * outputs.  MTP verify through the pool API (initial_state_indices) of sglang PR #23273, Summary; bf16
 * state, T beyond 4 and intermediate caching from its Requirements (FlashInfer #2679).
 */
GDN_API gdn_status gdn_mtp_verify(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                          const void* b, const float* A_log, const float* dt_bias, const void* state_pool,
                          const int32_t* state_indices, void* o, void* intermediate_states,
                          int32_t* err_word, gdn_stream_t stream);

/*
 * gdn_commit -- state_pool[state_indices[b], :] = intermediate_states[b, accept_len[b] - 1, :] (all heads),
 * bit for bit, for every active lane with accept_len[b] >= 1; accept_len 0 leaves the slot as it is.
 * Uses dims->B, T, HV, DK, DV, num_slots and state_dtype only.  The accepted-prefix checkpoint write of
 * the commit contract in TensorRT-LLM PR #20937 (GB300 Qwen3.8-Flash-Next NVFP4), "Moved out of this PR"
 * (the manager's all-layer commit) and its commit message, MTP > Verify (checkpoint-commit contract).
 */
GDN_API gdn_status gdn_commit(const gdn_dims* dims, void* state_pool, const int32_t* state_indices,
                      const void* intermediate_states, const int32_t* accept_len, int32_t* err_word,
                      gdn_stream_t stream);

/*
 * gdn_commit_replay -- the same pool update as gdn_commit, without intermediate states: for every active
 * lane with accept_len[b] >= 1, the first accept_len[b] tokens are run again from state_pool[slot] (which
 * gdn_mtp_verify left unchanged) and the final state is written back into that slot, rounded to
 * state_dtype.  fp32 state, or T > 8: the token-by-token arithmetic of gdn_mtp_verify, so the slot receives
 * exactly the bits gdn_commit would copy from intermediate_states[b, accept_len[b] - 1].  bf16 state with
 * T <= 8: the same state in chunked form (S_L = gamma S_0 + a sum of rank-1 terms, S_0 k on the tensor
 * cores with k split into bf16 hi + lo parts), within fp32-level error of that copy before the final bf16
 * rounding, so the two may differ in the last bf16 bit.  q, k, v, a, b, A_log, dt_bias, scale and l2_eps
 * must be those the verify call used; no outputs are written; accept_len 0 leaves the slot as it is,
 * lengths outside 0..T set GDN_ERRBIT_ACCEPT_LEN.  Verify then moves 1 state instead of 1 + T, at the cost
 * of reading each state once more here: the cached replay with in-kernel commit of TensorRT-LLM PR #20937
 * (GB300 Qwen3.8-Flash-Next NVFP4), "MTP > Verify" and "Moved out of this PR".
 */
GDN_API gdn_status gdn_commit_replay(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                             const void* b, const float* A_log, const float* dt_bias, void* state_pool,
                             const int32_t* state_indices, const int32_t* accept_len, int32_t* err_word,
                             gdn_stream_t stream);

/* The gated RMSNorm applied to a verify's outputs (gdn_mtp_verify_gated, gdn_mtp_verify_commit): exactly
 * gdn_gated_rmsnorm of the o the call stores,
 *     y[b,t,h,i] = o[b,t,h,i] / sqrt(mean_i(o[b,t,h,:]^2) + eps) * norm_weight[i] * silu(z[b,t,h,i]),
 * computed in fp32 and stored in out_dtype; rows of padded lanes are left untouched.  Device memory. */
typedef struct gdn_gated_norm_out {
    const void* z;             /* [B, T, HV, DV] z_dtype: the gate projection */
    int32_t z_dtype;           /* gdn_dtype of z */
    const float* norm_weight;  /* [DV] fp32 */
    float eps;                 /* finite, >= 0 */
    void* y;                   /* [B, T, HV, DV] out_dtype; may be o itself (then o is replaced by y) */
} gdn_gated_norm_out;

/*
 * gdn_mtp_verify_gated -- gdn_mtp_verify (o and, if given, intermediate_states, as that call writes them)
 * followed by the gated RMSNorm of o into norm->y.  Where the verify runs on the chunked kernel (a bf16 pool
 * without intermediate states, T <= 8, DK >= 64), the norm runs inside it while DV <= 128 and the batch leaves
 * each of its item pipelines one item at most, else gdn_gated_rmsnorm runs after it.  Elsewhere the token-by-token
 * kernels apply it in the same launch: the CTAs that share a head run as one thread-block cluster (at most 8, i.e.
 * DV <= 256, or DV <= 1024 where one CTA holds 128 rows) and meet their sums of squares in distributed shared
 * memory.  A wider head, or a grid of more CTAs than the GPU holds at once (where the two launches measured faster),
 * gets the norm's own launch.  The decode-rows gated norm of TensorRT-LLM PR #20937 (GB300
 * Qwen3.8-Flash-Next NVFP4), Per-File QA Perspective, Source files, fused into the recurrence's output.
 */
GDN_API gdn_status gdn_mtp_verify_gated(const gdn_dims* dims, const void* q, const void* k, const void* v,
                                        const void* a, const void* b, const float* A_log, const float* dt_bias,
                                        const void* state_pool, const int32_t* state_indices, void* o,
                                        void* intermediate_states, const gdn_gated_norm_out* norm, int32_t* err_word,
                                        gdn_stream_t stream);

/*
 * gdn_decode_gated -- gdn_decode (the outputs and the write-back as that call stores them) with the gated RMSNorm of
 * o into norm->y, in the same launch where the head's CTAs fit one cluster and the grid one wave (as in
 * gdn_mtp_verify_gated above), else followed by the norm's own launch.  The decode-rows gated norm of TensorRT-LLM PR #20937, Per-File QA
 * Perspective, Source files (gdn_decode_rows_gated_norm).  Arguments, errors and ownership as gdn_decode and
 * gdn_gated_norm_out.
 */
GDN_API gdn_status gdn_decode_gated(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                                    const void* b, const float* A_log, const float* dt_bias, void* state_pool,
                                    const int32_t* state_indices, void* o, const gdn_gated_norm_out* norm,
                                    int32_t* err_word, gdn_stream_t stream);

/* The tokens of an earlier gdn_mtp_verify call on the same lanes, whose accepted prefix gdn_mtp_verify_commit
 * commits before it verifies: the compact recovery record of a speculative step (its k, v, a, b and accept
 * lengths; q is not needed, the replay writes no outputs).  All device memory, layouts as in the header. */
typedef struct gdn_replay_tokens {
    int32_t T;                 /* tokens per lane of that call, 1 .. GDN_MAX_T */
    const void* k;             /* [B, T, HK, DK] qkv_dtype, 16-byte aligned */
    const void* v;             /* [B, T, HV, DV] qkv_dtype */
    const void* a;             /* [B, T, HV] qkv_dtype */
    const void* b;             /* [B, T, HV] qkv_dtype */
    const int32_t* accept_len; /* [B] int32: lane b commits its first accept_len[b] tokens (0: none) */
} gdn_replay_tokens;

/*
 * gdn_mtp_verify_commit -- one speculative step in one pass over the state pool: for every active lane, first
 * the commit of the earlier call's accepted prefix, exactly gdn_commit_replay(prev) (the state after
 * prev->accept_len[b] of prev's tokens written into state_pool[slot], rounded to state_dtype), then verify of
 * this call's T tokens from the slot as just written, exactly gdn_mtp_verify without intermediate states (o).
 * dims describes this call (dims->T tokens); prev->T may differ from it (the draft width may change between
 * steps).  With a bf16 pool, both token counts <= 4 and DK >= 64, one kernel reads each state once and writes it
 * once; otherwise the two calls run back to back (with more tokens they measured faster as two launches).  With
 * norm != NULL, the verify is gdn_mtp_verify_gated's (o and the gated norm into norm->y).  An accept length outside 0 .. prev->T sets
 * GDN_ERRBIT_ACCEPT_LEN and commits nothing for that lane (its verify still runs from the slot as it is).  The
 * in-kernel commit of TensorRT-LLM PR #20937 (GB300 Qwen3.8-Flash-Next NVFP4), "Moved out of this PR" (commits
 * in-kernel below 16 decode requests), fed by the compact GDN recovery records of the issue "Proposal: native
 * BF16 MTP speculative decoding for dense Qwen3.8-27B".
 */
GDN_API gdn_status gdn_mtp_verify_commit(const gdn_dims* dims, const gdn_replay_tokens* prev, const void* q,
                                         const void* k, const void* v, const void* a, const void* b,
                                         const float* A_log, const float* dt_bias, void* state_pool,
                                         const int32_t* state_indices, void* o, const gdn_gated_norm_out* norm,
                                         int32_t* err_word, gdn_stream_t stream);

/*
 * gdn_prefill -- prefill of B variable-length sequences packed along one token axis of N = dims->T tokens
 * (here T is the total token count, 0 .. 2^31 - 1, not bounded by GDN_MAX_T):
 *     q, k  [N, HK, DK]   v, o  [N, HV, DV]   a, b  [N, HV]   (qkv_dtype; o in out_dtype)
 *     cu_seqlens          [B + 1] int32, device: sequence b is tokens cu_seqlens[b] .. cu_seqlens[b+1]-1
 *     has_initial_state   [B] int32, device, nullable (NULL: every sequence has one)
 * Sequence b with slot = state_indices[b] != -1 starts from state_pool[slot, h] if has_initial_state[b]
 * is non-zero, else from the zero state (the slot is then not read: a fresh slot may hold anything), runs
 * its tokens with the recurrence above, writes o at their positions and the final state into
 * state_pool[slot, h], rounded to state_dtype once (the running state stays fp32).  An empty sequence
 * leaves its slot as it is.  Sequences must not overlap (their outputs would race); they may leave gaps
 * between them (o is not written there).  Bounds that are negative,
 * decreasing or beyond N skip the sequence and set GDN_ERRBIT_SEQLEN; a bad index sets GDN_ERRBIT_INDEX
 * (checked first).  Distinct active sequences must use distinct slots.  The chunked gated delta rule with
 * bf16 state pools and an initial-state mask ("fresh-state zeroing") of TensorRT-LLM PR #20937 (GB300
 * Qwen3.8-Flash-Next NVFP4), Per-File QA Perspective, Source files and Test-code files.  Alignment: q, k,
 * state_pool on 16 bytes, the rest on their element size.
 */
GDN_API gdn_status gdn_prefill(const gdn_dims* dims, const int32_t* cu_seqlens, const void* q, const void* k,
                               const void* v, const void* a, const void* b, const float* A_log,
                               const float* dt_bias, void* state_pool, const int32_t* state_indices,
                               const int32_t* has_initial_state, void* o, int32_t* err_word, gdn_stream_t stream);

/*
 * gdn_gated_rmsnorm -- gated RMSNorm of `rows` rows of DV outputs (one value head of one token per row):
 *     y[r, i] = o[r, i] / sqrt(mean_i(o[r, i]^2) + eps) * norm_weight[i] * silu(z[r, i]),
 *     silu(x) = x * sigmoid(x),
 * in fp32, y stored in o_dtype (round to nearest even for bf16).  o, y [rows, DV] o_dtype; z [rows, DV]
 * z_dtype (the gate projection); norm_weight [DV] fp32; all device memory.  y may be o itself (in place),
 * no other overlap.  rows == 0 enqueues nothing.  The decode-rows gated norm of TensorRT-LLM PR #20937,
 * Per-File QA Perspective, Source files (the page gives no formula: RMS over the value dimension, one
 * weight per column shared by all heads, SiLU gate after the norm, is the reading taken).  eps must be
 * finite and >= 0 (GDN_ERR_VALUE); o, z, y, norm_weight aligned to their element size.
 */
GDN_API gdn_status gdn_gated_rmsnorm(int64_t rows, int32_t DV, int32_t o_dtype, int32_t z_dtype, const void* o,
                                     const void* z, const float* norm_weight, float eps, void* y,
                                     gdn_stream_t stream);

/*
 * The in_proj projection of the decode / verify rows with its causal conv1d epilogue: TensorRT-LLM PR #20937
 * (GB300 Qwen3.8-Flash-Next NVFP4), What changes, Decode at small batch ("the in_proj GEMV with a fused conv1d
 * epilogue, for 2..16 verify rows and up to 8 decode rows").  The page gives no formula; the reading taken:
 *
 *   W [C, H] bf16 holds the C = 2*HK*DK + 2*HV*DV + 2*HV output channels in the order
 *     q (HK*DK) | k (HK*DK) | v (HV*DV) | z (HV*DV) | b (HV) | a (HV);
 *   the first Cc = 2*HK*DK + HV*DV channels (q, k, v) pass through a K-tap causal depthwise convolution whose
 *   state is the K-1 previous inputs of each channel, per pool slot:
 *     conv_state [num_slots, K-1, Cc] conv_dtype (oldest first),
 *   For lane b (rows b*T .. b*T+T-1 of x [B*T, H] bf16) with slot = state_indices[b] != -1, channel c, row t:
 *     p[t, c] = sum_h W[c, h] x[b*T + t, h]                      (fp32 accumulation)
 *     u[t, c] = p[t, c] rounded to conv_dtype                    (c < Cc: the value the state stores)
 *     seq     = conv_state[slot, 0 .. K-2, c], u[0 .. T-1, c]
 *     y[t, c] = conv_b[c] + sum_{j < K} conv_w[c, j] seq[t + j, c], then y * sigmoid(y) if dims->silu
 *   q, k [B, T, HK, DK], v [B, T, HV, DV] <- y of their channels; z [B, T, HV, DV], b, a [B, T, HV] <- p of theirs
 *   (all out_dtype).
 */
typedef struct gdn_conv_dims {
    int32_t B;          /* request lanes, 0 .. 65535 */
    int32_t T;          /* rows per lane, 1 .. GDN_MAX_T */
    int32_t H;          /* hidden size: a multiple of 8, 8 .. 65536 */
    int32_t HK;         /* query/key heads of the outputs, >= 1 */
    int32_t HV;         /* value heads, a multiple of HK */
    int32_t DK;         /* key dimension, >= 1 */
    int32_t DV;         /* value dimension, >= 1 */
    int32_t K;          /* convolution taps, 2 .. 4 */
    int32_t num_slots;  /* convolution-state slots, >= 1 */
    int32_t conv_dtype; /* gdn_dtype of conv_state and of the recovery records */
    int32_t out_dtype;  /* gdn_dtype of q, k, v, z, b, a */
    int32_t silu;       /* 1: SiLU after the convolution, 0: none */
} gdn_conv_dims;

/* Outputs of gdn_in_proj_conv: the inputs of gdn_decode / gdn_mtp_verify (q, k, v, a, b) and of the gated norm
 * (z); device memory, out_dtype, element-aligned, no overlap with anything else. */
typedef struct gdn_in_proj_out {
    void* q; /* [B, T, HK, DK] */
    void* k; /* [B, T, HK, DK] */
    void* v; /* [B, T, HV, DV] */
    void* z; /* [B, T, HV, DV] */
    void* b; /* [B, T, HV] */
    void* a; /* [B, T, HV] */
} gdn_in_proj_out;

/*
 * gdn_in_proj_conv -- the projection and convolution above for every lane whose index is not -1.
 * write_state = 1 (decode rows): conv_state[slot, j, c] = seq[T + j, c] for j < K-1 (the last K-1 entries).
 * write_state = 0 (verify rows): conv_state is only read; if records is not NULL it receives u:
 *     records [B, T, Cc] conv_dtype, the verify rows' recovery records for gdn_conv_commit.
 * conv_w [Cc, K] fp32, conv_b [Cc] fp32 or NULL (zero).  x and W start on 16 bytes; the rest on their element
 * size.  Lanes with index -1 are skipped (outputs, records and slot untouched); an index < -1 or >= num_slots
 * skips the lane and sets GDN_ERRBIT_INDEX.  Distinct active lanes must use distinct slots when write_state = 1.
 * The waits of the kernel on its own copies are bounded (GDN_ERRBIT_TIMEOUT, outputs of the tile left unwritten).
 */
GDN_API gdn_status gdn_in_proj_conv(const gdn_conv_dims* dims, const void* x, const void* W, const float* conv_w,
                                    const float* conv_b, void* conv_state, const int32_t* state_indices,
                                    int32_t write_state, const gdn_in_proj_out* out, void* records,
                                    int32_t* err_word, gdn_stream_t stream);

/*
 * gdn_conv_commit -- the convolution state after each lane's first L = accept_len[b] verify rows: with seq =
 * conv_state[slot, 0 .. K-2, c], records[b, 0 .. T-1, c], conv_state[slot, j, c] = seq[L + j, c] (bit copies).
 * L = 0 leaves the slot; L outside 0 .. T sets GDN_ERRBIT_ACCEPT_LEN, a bad index GDN_ERRBIT_INDEX (the lane is
 * skipped).  The commit of the convolution state with the accepted prefix (issue "Proposal: native BF16 MTP
 * speculative decoding for dense Qwen3.8-27B", What: the compact GDN recovery records and their commit).  Only
 * dims->B, T, HK, HV, DK, DV, K, num_slots and conv_dtype are read.
 */
GDN_API gdn_status gdn_conv_commit(const gdn_conv_dims* dims, void* conv_state, const int32_t* state_indices,
                                   const void* records, const int32_t* accept_len, int32_t* err_word,
                                   gdn_stream_t stream);

/* Static string naming a status; never NULL. */
GDN_API const char* gdn_status_string(gdn_status status);

/* cudaError_t of the calling thread's last GDN_ERR_CUDA (0 if none). */
GDN_API int32_t gdn_last_cuda_error(void);

/* ABI version of this header: 1. */
GDN_API int32_t gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
