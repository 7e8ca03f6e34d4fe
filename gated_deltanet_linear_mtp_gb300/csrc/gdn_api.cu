// gdn_api.cu -- the C ABI of libgdn.so (include/gdn.h): host-side validation, then one kernel launch on the
// caller's stream.  Every check that needs no device data happens here, before anything is enqueued, so a
// rejected call has no side effect.  No allocation, no synchronisation, no global mutable state (the last
// CUDA error is thread-local).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {

namespace {

thread_local int32_t g_last_cuda_error = 0;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_dtype(int32_t d) { return d == GDN_F32 || d == GDN_BF16; }

size_t dtype_bytes(int32_t d) { return d == GDN_F32 ? 4 : 2; }

bool supported_dk(int32_t dk) { return dk == 16 || dk == 32 || dk == 64 || dk == 128 || dk == 256; }

// Sizes common to every call.  `need_io`: q/k/v/o dtypes and the scalars matter (decode, verify).
// `prefill`: T is the total token count of the packed sequences (0 .. INT32_MAX), not tokens per lane.
gdn_status check_dims(const gdn_dims* d, bool need_io, bool prefill = false) {
    if (d == nullptr) return GDN_ERR_NULL;
    if (d->B < 0 || d->B > 65535) return GDN_ERR_SHAPE;
    if (prefill ? d->T < 0 : (d->T < 1 || d->T > GDN_MAX_T)) return GDN_ERR_SHAPE;
    if (d->HV < 1 || d->HV > 65535 || d->DV < 1 || d->num_slots < 1) return GDN_ERR_SHAPE;
    if (!valid_dtype(d->state_dtype)) return GDN_ERR_DTYPE;
    if (need_io) {
        if (d->HK < 1 || d->HV % d->HK != 0) return GDN_ERR_SHAPE;
        if (!valid_dtype(d->qkv_dtype) || !valid_dtype(d->out_dtype)) return GDN_ERR_DTYPE;
        if (!std::isfinite(d->scale) || !std::isfinite(d->l2_eps) || d->l2_eps < 0.f) return GDN_ERR_VALUE;
    }
    if (d->DK < 1) return GDN_ERR_SHAPE;
    if (!supported_dk(d->DK)) return GDN_ERR_UNSUPPORTED;
    // every element offset is formed in int64: bound the largest array (the cache) well inside it
    const double cache_elems = prefill ? (double)d->T * d->HV * (double)d->DV
                                       : (double)d->B * d->T * d->HV * (double)d->DV * d->DK;
    const double pool_elems = (double)d->num_slots * d->HV * (double)d->DV * d->DK;
    if (cache_elems > 4.0e18 || pool_elems > 4.0e18) return GDN_ERR_SHAPE;
    return GDN_OK;
}

// Sizes of gdn_in_proj_conv / gdn_conv_commit (`commit`: H, out_dtype and silu are not read).  Cc and C: the
// convolved and all output channels.  C is bounded so that a grid dimension (C / 128 tiles) and every element
// offset stay in range.
gdn_status check_conv_dims(const gdn_conv_dims* d, bool commit, int64_t* Cc, int64_t* C) {
    if (d == nullptr) return GDN_ERR_NULL;
    if (d->B < 0 || d->B > 65535 || d->T < 1 || d->T > GDN_MAX_T) return GDN_ERR_SHAPE;
    if (d->HK < 1 || d->HV < 1 || d->HV > 65535 || d->HV % d->HK != 0 || d->DK < 1 || d->DV < 1) return GDN_ERR_SHAPE;
    if (d->K < 2 || d->K > 4 || d->num_slots < 1) return GDN_ERR_SHAPE;
    if (!valid_dtype(d->conv_dtype)) return GDN_ERR_DTYPE;
    if (!commit) {
        if (d->H < 8 || d->H > 65536 || d->H % 8 != 0) return GDN_ERR_SHAPE;
        if (!valid_dtype(d->out_dtype)) return GDN_ERR_DTYPE;
        if (d->silu != 0 && d->silu != 1) return GDN_ERR_VALUE;
    }
    const int64_t qk = (int64_t)d->HK * d->DK, vz = (int64_t)d->HV * d->DV;
    if (qk > (1 << 22) || vz > (1 << 22)) return GDN_ERR_SHAPE;
    *Cc = 2 * qk + vz;
    *C = *Cc + vz + 2 * (int64_t)d->HV;
    if (*C > (int64_t)65535 * 128) return GDN_ERR_SHAPE;
    if ((double)d->num_slots * (d->K - 1) * (double)*Cc > 4.0e18) return GDN_ERR_SHAPE;
    return GDN_OK;
}

// `o` may be NULL only where the call has no outputs (replay commit: need_o = false).
gdn_status check_io(const gdn_dims* d, const void* q, const void* k, const void* v, const void* a, const void* b,
                    const float* A_log, const float* dt_bias, const void* pool, const int32_t* idx, const void* o,
                    const int32_t* err, bool need_o = true) {
    if (!q || !k || !v || !a || !b || !A_log || !dt_bias || !pool || !idx || (need_o && !o)) return GDN_ERR_NULL;
    const uintptr_t in_sz = dtype_bytes(d->qkv_dtype);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(pool, 16)) return GDN_ERR_ALIGN;
    if (!aligned(v, in_sz) || !aligned(a, in_sz) || !aligned(b, in_sz)) return GDN_ERR_ALIGN;
    if (!aligned(A_log, 4) || !aligned(dt_bias, 4) || !aligned(idx, 4)) return GDN_ERR_ALIGN;
    if (!aligned(o, dtype_bytes(d->out_dtype))) return GDN_ERR_ALIGN;
    if (err && !aligned(err, 4)) return GDN_ERR_ALIGN;
    return GDN_OK;
}

gdn_status finish(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    g_last_cuda_error = (int32_t)e;
    return GDN_ERR_CUDA;
}

RecurrentParams make_params(const gdn_dims* d, const void* q, const void* k, const void* v, const void* a,
                            const void* b, const float* A_log, const float* dt_bias, const void* pool_in,
                            void* pool_out, const int32_t* idx, const int32_t* steps, void* o, void* cache,
                            int32_t* err) {
    RecurrentParams p{};  // the replay-commit + verify fields stay null unless set by that call
    p.q = q;
    p.k = k;
    p.v = v;
    p.a = a;
    p.b = b;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.pool_in = pool_in;
    p.pool_out = pool_out;
    p.indices = idx;
    p.steps = steps;
    p.o = o;
    p.cache = cache;
    p.err = err;
    p.T = d->T;
    p.HK = d->HK;
    p.HV = d->HV;
    p.DV = d->DV;
    p.num_slots = d->num_slots;
    p.out_bf16 = d->out_dtype == GDN_BF16;
    p.v_vec = aligned(v, 16) && ((int64_t)d->DV * (int64_t)dtype_bytes(d->qkv_dtype)) % 16 == 0;
    p.scale = d->scale;
    p.l2_eps = d->l2_eps;
    return p;
}

gdn_status run_recurrent(const gdn_dims* d, const void* q, const void* k, const void* v, const void* a,
                         const void* b, const float* A_log, const float* dt_bias, const void* pool_in,
                         void* pool_out, const int32_t* idx, const int32_t* steps, void* o, void* cache,
                         int32_t* err, cudaStream_t stream) {
    const RecurrentParams p =
        make_params(d, q, k, v, a, b, A_log, dt_bias, pool_in, pool_out, idx, steps, o, cache, err);
    const bool qkv_bf16 = d->qkv_dtype == GDN_BF16;
    if (d->state_dtype == GDN_F32) return finish(launch_recurrent_f32state(p, d->B, d->DK, qkv_bf16, stream));
    return finish(launch_recurrent_bf16state(p, d->B, d->DK, qkv_bf16, stream));
}

// The gated norm of a verify's outputs: its record checked; `fused` is set when the chunked kernel applies it
// (a bf16 pool without intermediate states, the kernel's range, DV <= 128: one item holds a whole head).
gdn_status check_norm(const gdn_dims* d, const gdn_gated_norm_out* n, const void* o) {
    if (n == nullptr) return GDN_OK;
    if (!n->z || !n->norm_weight || !n->y) return GDN_ERR_NULL;
    if (!valid_dtype(n->z_dtype)) return GDN_ERR_DTYPE;
    if (!std::isfinite(n->eps) || n->eps < 0.f) return GDN_ERR_VALUE;
    if (!aligned(n->z, dtype_bytes(n->z_dtype)) || !aligned(n->y, dtype_bytes(d->out_dtype)) ||
        !aligned(n->norm_weight, 4))
        return GDN_ERR_ALIGN;
    (void)o;
    return GDN_OK;
}

// Inside the chunked kernel the norm lengthens every item's chain, which paid only while each group of the GPU
// has at most one item (verify T=4, HV=32: fused 14.3 vs 14.9 us at B <= 4, slower from B = 16 up, where the
// separate norm launch overlaps better): fused then, a norm launch otherwise.
bool norm_fused(const gdn_dims* d, bool cache) {
    if (d->state_dtype != GDN_BF16 || cache || d->DV > 128 ||
        !chunked_verify_eligible(d->B, d->T, d->DK, d->DV, d->HV, d->num_slots))
        return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    return (int64_t)d->B * d->HV <= (int64_t)sms * kChunkGroupsPerSm;
}

void set_norm(RecurrentParams& p, const gdn_gated_norm_out* n) {
    p.nz = n->z;
    p.nz_bf16 = n->z_dtype == GDN_BF16;
    p.nw = n->norm_weight;
    p.ny = n->y;
    p.neps = n->eps;
    p.nz_vec = p.DV % 8 == 0 && aligned(n->z, 16);
}

// the standalone norm of the stored o, rows of padded or invalid lanes left untouched
gdn_status run_norm(const gdn_dims* d, const gdn_gated_norm_out* n, const void* o, const int32_t* idx,
                    cudaStream_t st) {
    GatedNormParams g{};
    g.o = o;
    g.z = n->z;
    g.w = n->norm_weight;
    g.y = n->y;
    g.rows = (int64_t)d->B * d->T * d->HV;
    g.DV = d->DV;
    g.o_bf16 = d->out_dtype == GDN_BF16;
    g.z_bf16 = n->z_dtype == GDN_BF16;
    g.vec = d->DV % 8 == 0 && aligned(o, 16) && aligned(n->z, 16) && aligned(n->y, 16) && aligned(n->norm_weight, 16);
    g.eps = n->eps;
    g.lane_slot = idx;
    g.rows_per_lane = (int64_t)d->T * d->HV;
    g.num_slots = d->num_slots;
    return finish(launch_gated_norm(g, st));
}

gdn_status verify_commit(const gdn_dims* dims, const gdn_replay_tokens* prev, const void* q, const void* k,
                         const void* v, const void* a, const void* b, const float* A_log, const float* dt_bias,
                         void* state_pool, const int32_t* state_indices, void* o, const gdn_gated_norm_out* norm,
                         int32_t* err_word, gdn_stream_t stream) {
    gdn_status s = check_dims(dims, true);
    if (s != GDN_OK) return s;
    if (prev == nullptr) return GDN_ERR_NULL;
    if (prev->T < 1 || prev->T > GDN_MAX_T) return GDN_ERR_SHAPE;
    gdn_dims pd = *dims;  // the earlier call's shape: its own token count
    pd.T = prev->T;
    s = check_dims(&pd, true);
    if (s != GDN_OK) return s;
    if (dims->B == 0) return GDN_OK;
    s = check_io(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word);
    if (s != GDN_OK) return s;
    // the earlier tokens have the layouts of k, v, a, b (no q: the replay writes no outputs)
    s = check_io(&pd, prev->k, prev->k, prev->v, prev->a, prev->b, A_log, dt_bias, state_pool, state_indices, nullptr,
                 err_word, false);
    if (s != GDN_OK) return s;
    if (!prev->accept_len) return GDN_ERR_NULL;
    if (!aligned(prev->accept_len, 4)) return GDN_ERR_ALIGN;
    s = check_norm(dims, norm, o);
    if (s != GDN_OK) return s;
    if (norm && (double)dims->B * dims->T * dims->HV > (double)gated_norm_max_rows()) return GDN_ERR_SHAPE;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dims->state_dtype == GDN_BF16 && (norm == nullptr || norm_fused(dims, false))) {
        RecurrentParams p = make_params(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_pool, state_indices,
                                        prev->accept_len, o, nullptr, err_word);
        p.rk = prev->k;
        p.rv = prev->v;
        p.ra = prev->a;
        p.rb = prev->b;
        p.rT = prev->T;
        if (norm) set_norm(p, norm);
        cudaError_t e = cudaSuccess;
        if (launch_replay_verify_bf16state(p, dims->B, dims->DK, dims->qkv_dtype == GDN_BF16, st, e)) return finish(e);
    }
    // outside the one-pass kernel's range: the same two steps as two launches, the replay commit (q is not read
    // for outputs; the earlier k stands in for it) and then the verify from the committed slots
    s = run_recurrent(&pd, prev->k, prev->k, prev->v, prev->a, prev->b, A_log, dt_bias, state_pool, state_pool,
                      state_indices, prev->accept_len, nullptr, nullptr, err_word, st);
    if (s != GDN_OK) return s;
    if (norm == nullptr)
        return run_recurrent(dims, q, k, v, a, b, A_log, dt_bias, state_pool, nullptr, state_indices, nullptr, o,
                             nullptr, err_word, st);
    return gdn_mtp_verify_gated(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, nullptr, norm,
                                err_word, stream);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_decode(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                      const void* b, const float* A_log, const float* dt_bias, void* state_pool,
                      const int32_t* state_indices, void* o, int32_t* err_word, gdn_stream_t stream) {
    gdn_status s = check_dims(dims, true);
    if (s != GDN_OK) return s;
    if (dims->B == 0) return GDN_OK;
    s = check_io(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word);
    if (s != GDN_OK) return s;
    return run_recurrent(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_pool, state_indices, nullptr, o,
                         nullptr, err_word, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_mtp_verify(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                          const void* b, const float* A_log, const float* dt_bias, const void* state_pool,
                          const int32_t* state_indices, void* o, void* intermediate_states,
                          int32_t* err_word, gdn_stream_t stream) {
    gdn_status s = check_dims(dims, true);
    if (s != GDN_OK) return s;
    if (dims->B == 0) return GDN_OK;
    s = check_io(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word);
    if (s != GDN_OK) return s;
    if (intermediate_states && !aligned(intermediate_states, 16)) return GDN_ERR_ALIGN;
    return run_recurrent(dims, q, k, v, a, b, A_log, dt_bias, state_pool, nullptr, state_indices, nullptr, o,
                         intermediate_states, err_word, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_commit(const gdn_dims* dims, void* state_pool, const int32_t* state_indices,
                      const void* intermediate_states, const int32_t* accept_len, int32_t* err_word,
                      gdn_stream_t stream) {
    gdn_status s = check_dims(dims, false);
    if (s != GDN_OK) return s;
    if (dims->B == 0) return GDN_OK;
    if (!state_pool || !state_indices || !intermediate_states || !accept_len) return GDN_ERR_NULL;
    if (!aligned(state_pool, 16) || !aligned(intermediate_states, 16)) return GDN_ERR_ALIGN;
    if (!aligned(state_indices, 4) || !aligned(accept_len, 4) || (err_word && !aligned(err_word, 4)))
        return GDN_ERR_ALIGN;
    CommitParams p;
    p.pool = state_pool;
    p.indices = state_indices;
    p.cache = intermediate_states;
    p.accept_len = accept_len;
    p.err = err_word;
    p.T = dims->T;
    p.num_slots = dims->num_slots;
    p.lane_bytes = (int64_t)dims->HV * dims->DV * dims->DK * (int64_t)dtype_bytes(dims->state_dtype);
    return finish(launch_commit(p, dims->B, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_commit_replay(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                             const void* b, const float* A_log, const float* dt_bias, void* state_pool,
                             const int32_t* state_indices, const int32_t* accept_len, int32_t* err_word,
                             gdn_stream_t stream) {
    gdn_status s = check_dims(dims, true);
    if (s != GDN_OK) return s;
    if (dims->B == 0) return GDN_OK;
    s = check_io(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, nullptr, err_word, false);
    if (s != GDN_OK) return s;
    if (!accept_len) return GDN_ERR_NULL;
    if (!aligned(accept_len, 4)) return GDN_ERR_ALIGN;
    return run_recurrent(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_pool, state_indices, accept_len,
                         nullptr, nullptr, err_word, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_mtp_verify_gated(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                                const void* b, const float* A_log, const float* dt_bias, const void* state_pool,
                                const int32_t* state_indices, void* o, void* intermediate_states,
                                const gdn_gated_norm_out* norm, int32_t* err_word, gdn_stream_t stream) {
    gdn_status s = check_dims(dims, true);
    if (s != GDN_OK) return s;
    if (norm == nullptr) return GDN_ERR_NULL;
    s = check_norm(dims, norm, o);
    if (s != GDN_OK) return s;
    if (dims->B == 0) return GDN_OK;
    if ((double)dims->B * dims->T * dims->HV > (double)gated_norm_max_rows()) return GDN_ERR_SHAPE;
    s = check_io(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word);
    if (s != GDN_OK) return s;
    if (intermediate_states && !aligned(intermediate_states, 16)) return GDN_ERR_ALIGN;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    RecurrentParams p = make_params(dims, q, k, v, a, b, A_log, dt_bias, state_pool, nullptr, state_indices, nullptr, o,
                                    intermediate_states, err_word);
    // the chunked kernel takes the norm when norm_fused says so, else a norm launch follows it; the token-by-token
    // kernels take it themselves (in the same launch, a cluster per head, or with their own norm launch)
    const bool chunked = dims->state_dtype == GDN_BF16 && intermediate_states == nullptr &&
                         chunked_verify_eligible(dims->B, dims->T, dims->DK, dims->DV, dims->HV, dims->num_slots);
    const bool fused = norm_fused(dims, intermediate_states != nullptr);
    if (fused || !chunked) set_norm(p, norm);
    const bool qkv_bf16 = dims->qkv_dtype == GDN_BF16;
    s = finish(dims->state_dtype == GDN_F32 ? launch_recurrent_f32state(p, dims->B, dims->DK, qkv_bf16, st)
                                            : launch_recurrent_bf16state(p, dims->B, dims->DK, qkv_bf16, st));
    if (s != GDN_OK || fused || !chunked) return s;
    return run_norm(dims, norm, o, state_indices, st);
}

gdn_status gdn_decode_gated(const gdn_dims* dims, const void* q, const void* k, const void* v, const void* a,
                            const void* b, const float* A_log, const float* dt_bias, void* state_pool,
                            const int32_t* state_indices, void* o, const gdn_gated_norm_out* norm, int32_t* err_word,
                            gdn_stream_t stream) {
    gdn_status s = check_dims(dims, true);
    if (s != GDN_OK) return s;
    if (norm == nullptr) return GDN_ERR_NULL;
    s = check_norm(dims, norm, o);
    if (s != GDN_OK) return s;
    if (dims->B == 0) return GDN_OK;
    if ((double)dims->B * dims->T * dims->HV > (double)gated_norm_max_rows()) return GDN_ERR_SHAPE;
    s = check_io(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word);
    if (s != GDN_OK) return s;
    RecurrentParams p = make_params(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_pool, state_indices, nullptr,
                                    o, nullptr, err_word);
    set_norm(p, norm);
    const bool qkv_bf16 = dims->qkv_dtype == GDN_BF16;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return finish(dims->state_dtype == GDN_F32 ? launch_recurrent_f32state(p, dims->B, dims->DK, qkv_bf16, st)
                                               : launch_recurrent_bf16state(p, dims->B, dims->DK, qkv_bf16, st));
}

gdn_status gdn_mtp_verify_commit(const gdn_dims* dims, const gdn_replay_tokens* prev, const void* q, const void* k,
                                 const void* v, const void* a, const void* b, const float* A_log, const float* dt_bias,
                                 void* state_pool, const int32_t* state_indices, void* o,
                                 const gdn_gated_norm_out* norm, int32_t* err_word, gdn_stream_t stream) {
    return verify_commit(dims, prev, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, norm, err_word,
                         stream);
}

gdn_status gdn_prefill(const gdn_dims* dims, const int32_t* cu_seqlens, const void* q, const void* k, const void* v,
                       const void* a, const void* b, const float* A_log, const float* dt_bias, void* state_pool,
                       const int32_t* state_indices, const int32_t* has_initial_state, void* o, int32_t* err_word,
                       gdn_stream_t stream) {
    gdn_status s = check_dims(dims, true, true);
    if (s != GDN_OK) return s;
    if (dims->B == 0 || dims->T == 0) return GDN_OK;
    s = check_io(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, o, err_word);
    if (s != GDN_OK) return s;
    if (!cu_seqlens) return GDN_ERR_NULL;
    if (!aligned(cu_seqlens, 4) || (has_initial_state && !aligned(has_initial_state, 4))) return GDN_ERR_ALIGN;
    const RecurrentParams p = make_params(dims, q, k, v, a, b, A_log, dt_bias, state_pool, state_pool, state_indices,
                                          nullptr, o, nullptr, err_word);
    return finish(launch_prefill(p, cu_seqlens, has_initial_state, dims->B, dims->T, dims->DK,
                                 dims->qkv_dtype == GDN_BF16, dims->state_dtype == GDN_BF16,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_gated_rmsnorm(int64_t rows, int32_t DV, int32_t o_dtype, int32_t z_dtype, const void* o, const void* z,
                             const float* norm_weight, float eps, void* y, gdn_stream_t stream) {
    if (rows < 0 || DV < 1 || rows > gated_norm_max_rows()) return GDN_ERR_SHAPE;
    if ((double)rows * DV > 4.0e18) return GDN_ERR_SHAPE;
    if (!valid_dtype(o_dtype) || !valid_dtype(z_dtype)) return GDN_ERR_DTYPE;
    if (!std::isfinite(eps) || eps < 0.f) return GDN_ERR_VALUE;
    if (rows == 0) return GDN_OK;
    if (!o || !z || !norm_weight || !y) return GDN_ERR_NULL;
    const uintptr_t osz = dtype_bytes(o_dtype), zsz = dtype_bytes(z_dtype);
    if (!aligned(o, osz) || !aligned(y, osz) || !aligned(z, zsz) || !aligned(norm_weight, 4)) return GDN_ERR_ALIGN;
    GatedNormParams p{};
    p.o = o;
    p.z = z;
    p.w = norm_weight;
    p.y = y;
    p.rows = rows;
    p.DV = DV;
    p.o_bf16 = o_dtype == GDN_BF16;
    p.z_bf16 = z_dtype == GDN_BF16;
    p.vec = DV % 8 == 0 && aligned(o, 16) && aligned(z, 16) && aligned(y, 16) && aligned(norm_weight, 16);
    p.eps = eps;
    return finish(launch_gated_norm(p, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_in_proj_conv(const gdn_conv_dims* dims, const void* x, const void* W, const float* conv_w,
                            const float* conv_b, void* conv_state, const int32_t* state_indices, int32_t write_state,
                            const gdn_in_proj_out* out, void* records, int32_t* err_word, gdn_stream_t stream) {
    int64_t Cc = 0, C = 0;
    gdn_status s = check_conv_dims(dims, false, &Cc, &C);
    if (s != GDN_OK) return s;
    if (write_state != 0 && write_state != 1) return GDN_ERR_VALUE;
    if (dims->B == 0) return GDN_OK;
    if (!x || !W || !conv_w || !conv_state || !state_indices || !out) return GDN_ERR_NULL;
    if (!out->q || !out->k || !out->v || !out->z || !out->b || !out->a) return GDN_ERR_NULL;
    const uintptr_t ssz = dtype_bytes(dims->conv_dtype), osz = dtype_bytes(dims->out_dtype);
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(conv_w, 4) || (conv_b && !aligned(conv_b, 4))) return GDN_ERR_ALIGN;
    if (!aligned(conv_state, ssz) || (records && !aligned(records, ssz)) || !aligned(state_indices, 4)) return GDN_ERR_ALIGN;
    if (!aligned(out->q, osz) || !aligned(out->k, osz) || !aligned(out->v, osz) || !aligned(out->z, osz) ||
        !aligned(out->b, osz) || !aligned(out->a, osz))
        return GDN_ERR_ALIGN;
    if (err_word && !aligned(err_word, 4)) return GDN_ERR_ALIGN;
    InProjConvParams p{};
    p.B = dims->B;
    p.T = dims->T;
    p.H = dims->H;
    p.HK = dims->HK;
    p.HV = dims->HV;
    p.DK = dims->DK;
    p.DV = dims->DV;
    p.K = dims->K;
    p.num_slots = dims->num_slots;
    p.Cc = Cc;
    p.C = C;
    p.conv_w = conv_w;
    p.conv_b = conv_b;
    p.state = conv_state;
    p.state_bf16 = dims->conv_dtype == GDN_BF16;
    p.state_vec = Cc % 8 == 0 && aligned(conv_state, 16);
    p.indices = state_indices;
    p.write_state = write_state;
    p.q = out->q;
    p.k = out->k;
    p.v = out->v;
    p.z = out->z;
    p.bo = out->b;
    p.ao = out->a;
    p.out_bf16 = dims->out_dtype == GDN_BF16;
    p.records = records;
    p.x = x;
    p.W = W;
    p.err = err_word;
    p.silu = dims->silu;
    return finish(launch_in_proj_conv(p, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_conv_commit(const gdn_conv_dims* dims, void* conv_state, const int32_t* state_indices,
                           const void* records, const int32_t* accept_len, int32_t* err_word, gdn_stream_t stream) {
    int64_t Cc = 0, C = 0;
    gdn_status s = check_conv_dims(dims, true, &Cc, &C);
    if (s != GDN_OK) return s;
    if (dims->B == 0) return GDN_OK;
    if (!conv_state || !state_indices || !records || !accept_len) return GDN_ERR_NULL;
    const uintptr_t ssz = dtype_bytes(dims->conv_dtype);
    if (!aligned(conv_state, ssz) || !aligned(records, ssz) || !aligned(state_indices, 4) || !aligned(accept_len, 4))
        return GDN_ERR_ALIGN;
    if (err_word && !aligned(err_word, 4)) return GDN_ERR_ALIGN;
    ConvCommitParams p{};
    p.state = conv_state;
    p.indices = state_indices;
    p.records = records;
    p.accept_len = accept_len;
    p.err = err_word;
    p.B = dims->B;
    p.T = dims->T;
    p.K = dims->K;
    p.num_slots = dims->num_slots;
    p.state_bf16 = dims->conv_dtype == GDN_BF16;
    p.Cc = Cc;
    return finish(launch_conv_commit(p, reinterpret_cast<cudaStream_t>(stream)));
}

const char* gdn_status_string(gdn_status status) {
    switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_NULL: return "GDN_ERR_NULL: a required pointer is NULL";
    case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE: a size is out of range or inconsistent";
    case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE: unknown dtype code";
    case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN: a pointer is misaligned";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: DK must be 16, 32, 64, 128 or 256";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: kernel launch failed (see gdn_last_cuda_error)";
    case GDN_ERR_VALUE: return "GDN_ERR_VALUE: scale or an epsilon not finite, or an epsilon < 0";
    }
    return "unknown gdn_status";
}

int32_t gdn_last_cuda_error(void) { return g_last_cuda_error; }

int32_t gdn_abi_version(void) { return 1; }

}  // extern "C"
