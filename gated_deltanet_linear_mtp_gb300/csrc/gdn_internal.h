// gdn_internal.h -- launch parameters shared by the C-ABI layer (gdn_api.cu) and the kernel translation
// units.  Not installed; the public interface is include/gdn.h.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace gdn {

// Decode, verify and replay commit share one kernel: decode writes the final state back (pool_out ==
// pool_in); verify optionally stores every intermediate state (cache != nullptr) and never writes the
// pool; replay commit runs steps[b] tokens per lane, writes no outputs and writes the state back.
struct RecurrentParams {
    const void* q;
    const void* k;
    const void* v;
    const void* a;
    const void* b;
    const float* A_log;
    const float* dt_bias;
    const void* pool_in;
    void* pool_out;  // nullptr: no write-back (verify)
    const int32_t* indices;
    const int32_t* steps;  // nullptr: T tokens per lane; else steps[b] in 0..T (replay commit)
    void* o;               // nullptr: no outputs (replay commit)
    void* cache;           // nullptr: no intermediate states
    int32_t* err;    // nullable
    int T, HK, HV, DV, num_slots;
    int out_bf16;
    int v_vec;  // v starts on 16 bytes and DV * sizeof(v) % 16 == 0: v is read in 16-byte chunks
    float scale, l2_eps;
    // replay commit + verify: the earlier call's tokens to commit first (rT per lane; steps[b] of them), with
    // q .. b above the tokens to verify; nullptr / 0 otherwise
    int rT;
    const void* rk;
    const void* rv;
    const void* ra;
    const void* rb;
    // gated RMSNorm of the stored o (the chunked verify's and the token-by-token kernels' epilogue): y = o /
    // sqrt(mean(o^2) + neps) * nw * silu(nz) per (token, head) row of DV, y in o's type; nz == nullptr: none
    const void* nz;
    const float* nw;
    void* ny;
    float neps;
    int nz_bf16;
    int nz_vec;  // z starts on 16 bytes and DV % 8 == 0: z is gathered in 16-byte chunks
};

struct CommitParams {
    void* pool;
    const int32_t* indices;
    const void* cache;
    const int32_t* accept_len;
    int32_t* err;
    int T, num_slots;
    int64_t lane_bytes;  // HV * DV * DK * element size: one lane's state, all heads
};

// The in_proj projection with its causal conv1d epilogue (gdn_in_proj_conv), and the convolution state's commit.
struct InProjConvParams {
    int B, T, H, HK, HV, DK, DV, K, num_slots;
    int64_t Cc, C;          // convolved channels (q | k | v), all channels (q | k | v | z | b | a)
    const float* conv_w;    // [Cc, K]
    const float* conv_b;    // [Cc] or nullptr
    void* state;            // [num_slots, K - 1, Cc]
    int state_bf16;
    int state_vec;          // state on 16 bytes and Cc % 8 == 0: its rows are gathered in 16-byte pieces
    const int32_t* indices;
    int write_state;        // decode: the last K - 1 entries of each lane's sequence go back to its slot
    void* q;                // [B, T, HK, DK]
    void* k;
    void* v;                // [B, T, HV, DV]
    void* z;
    void* bo;               // [B, T, HV]
    void* ao;
    int out_bf16;
    void* records;          // [B, T, Cc] state type, or nullptr
    const void* x;          // [B * T, H] bf16
    const void* W;          // [C, H] bf16
    int32_t* err;
    int silu;
};

struct ConvCommitParams {
    void* state;            // [num_slots, K - 1, Cc]
    const int32_t* indices;
    const void* records;    // [B, T, Cc]
    const int32_t* accept_len;
    int32_t* err;
    int B, T, K, num_slots, state_bf16;
    int64_t Cc;
};

struct GatedNormParams {
    const void* o;   // [rows, DV], o_bf16 ? bf16 : fp32
    const void* z;   // [rows, DV], z_bf16 ? bf16 : fp32
    const float* w;  // [DV]
    void* y;         // [rows, DV], o's type; may be o itself
    int64_t rows;
    int DV;
    int o_bf16, z_bf16;
    int vec;  // DV % 8 == 0 and o, z, y, w start on 16 bytes: 8 columns per access
    float eps;
    // rows of padded or invalid lanes left untouched: row r belongs to lane r / rows_per_lane, skipped when
    // lane_slot[lane] is outside 0 .. num_slots - 1; nullptr: every row
    const int32_t* lane_slot;
    int64_t rows_per_lane;
    int num_slots;
};

cudaError_t launch_recurrent_f32state(const RecurrentParams& p, int B, int DK, bool qkv_bf16, cudaStream_t s);
// A verify without intermediate states on a bf16 pool runs the chunked tensor-core kernel (which can also apply
// the gated norm when DV <= 128) when this holds.
bool chunked_verify_eligible(int B, int T, int DK, int DV, int HV, int num_slots);
constexpr int kChunkGroupsPerSm = 3;  // item pipelines of the chunked verify kernel per SM (DK <= 128)
cudaError_t launch_recurrent_bf16state(const RecurrentParams& p, int B, int DK, bool qkv_bf16, cudaStream_t s);
// Replay commit of p.rk .. p.rb (p.rT tokens per lane, p.steps[b] of them) and then verify of p.q .. p.b (p.T
// tokens) in one pass of the chunked kernel; false (nothing launched) when the call is outside that kernel's
// range (T or rT above 8, DK below 64, too many heads or items), else `err` is the launch's status.
bool launch_replay_verify_bf16state(const RecurrentParams& p, int B, int DK, bool qkv_bf16, cudaStream_t s,
                                    cudaError_t& err);
cudaError_t launch_commit(const CommitParams& p, int B, cudaStream_t s);
// prefill: p.T unused; the token axis has n_tokens entries, sequence b spans cu_seqlens[b] .. cu_seqlens[b+1]-1
cudaError_t launch_prefill(const RecurrentParams& p, const int32_t* cu_seqlens, const int32_t* has_init, int B,
                           int n_tokens, int DK, bool qkv_bf16, bool state_bf16, cudaStream_t s);
// prefill in chunked form on the tensor cores (gdn_prefill_chunked.cu): DK = 64 or 128
bool prefill_chunked_eligible(int DK);
cudaError_t launch_prefill_chunked(const RecurrentParams& p, const int32_t* cu_seqlens, const int32_t* has_init, int B,
                                   int n_tokens, int DK, bool qkv_bf16, bool state_bf16, cudaStream_t s);
cudaError_t launch_gated_norm(const GatedNormParams& p, cudaStream_t s);

// gdn_in_proj_conv.cu
cudaError_t launch_in_proj_conv(const InProjConvParams& p, cudaStream_t s);
cudaError_t launch_conv_commit(const ConvCommitParams& p, cudaStream_t s);
int64_t gated_norm_max_rows();

}  // namespace gdn
