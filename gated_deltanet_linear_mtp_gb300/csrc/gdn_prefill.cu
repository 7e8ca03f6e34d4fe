// gdn_prefill.cu -- prefill of packed variable-length sequences into the state pool (sm_103a).
//
// Sequence b owns tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 of q, k [N, HK, DK], v, o [N, HV, DV] and a, b
// [N, HV].  It starts from state_pool[state_indices[b], h] (or from zero when has_initial_state[b] == 0:
// the slot is then never read), runs every token, writes o at its positions and the final state back into
// the slot.  The chunked gated delta rule with bf16 state pools and an initial-state mask ("fresh-state
// zeroing") of TensorRT-LLM PR #20937, Per-File QA Perspective, Source files and Test-code files.
//
// Form: the token-by-token (rank-1) update of gdn_recurrent.cuh (lane layout, token prologue, token loop).
// One CTA of 4 warps holds a block of RPC = Split<DK>::RPC rows of one (sequence, value head) in fp32
// registers for the whole sequence; the tokens go through shared memory in chunks of CT (one pass of
// TokenPrologue), double-buffered: the loads of chunk c+1 are in flight in registers while chunk c runs,
// and are normalised into the other buffer after it.  The state is rounded to the pool's type once, at the
// final write-back.  6 CTAs per SM (80 registers, no spills) measured faster than 7 (72, spilling).
#include "gdn_recurrent.cuh"

namespace gdn {

template <int DK>
struct PrefillPlan {
    using SP = Split<DK>;
    // token layout of the prologue does not depend on the input type
    using Pro = TokenPrologue<DK, float, SP::RPC, SP::THREADS>;
    static constexpr int CT = Pro::TPASS < 16 ? Pro::TPASS : 16;  // tokens per chunk
    // one buffer: q [CT][DK], k [CT][DK], v [CT][RPC], g, beta, kh.qh [CT]; a 16-byte multiple
    static constexpr size_t BUF_FLOATS = ((size_t)2 * CT * DK + (size_t)CT * SP::RPC + 3 * CT + 3) & ~(size_t)3;
    static constexpr size_t SMEM_BYTES = 2 * sizeof(float) * BUF_FLOATS;
    static constexpr int MIN_CTAS = Split<DK>::MIN_CTAS_PER_SM;
};

// Point the token inputs (q, k, v, a, b) of `c` at the chunk of `len` tokens starting at token `tok`, so that
// lane 0 of the [B, T] indexing of the token prologue addresses it (T = len).  The outputs are set apart
// (chunk_outputs): the prologue of the next chunk and the token loop of this one run on the same struct.
template <int DK, typename InT>
__device__ __forceinline__ void chunk_inputs(RecurrentParams& c, const RecurrentParams& p, int64_t tok, int len) {
    c.q = static_cast<const InT*>(p.q) + tok * p.HK * DK;
    c.k = static_cast<const InT*>(p.k) + tok * p.HK * DK;
    c.v = static_cast<const InT*>(p.v) + tok * p.HV * p.DV;
    c.a = static_cast<const InT*>(p.a) + tok * p.HV;
    c.b = static_cast<const InT*>(p.b) + tok * p.HV;
    c.T = len;
}

// o of the chunk starting at token `tok`; the pool write-back (run_tokens) only after the sequence's last chunk
__device__ __forceinline__ void chunk_outputs(RecurrentParams& c, const RecurrentParams& p, int64_t tok, bool last) {
    if (p.out_bf16)
        c.o = static_cast<__nv_bfloat16*>(p.o) + tok * p.HV * p.DV;
    else
        c.o = static_cast<float*>(p.o) + tok * p.HV * p.DV;
    c.pool_out = last ? p.pool_out : nullptr;
}

template <int DK, typename InT, typename StT>
__global__ void __launch_bounds__(Split<DK>::THREADS, PrefillPlan<DK>::MIN_CTAS)
    gdn_prefill_kernel(const RecurrentParams p, const int32_t* __restrict__ cu_seqlens,
                       const int32_t* __restrict__ has_init, int n_tokens) {
    using SP = Split<DK>;
    using SL = Slice8<StT>;
    using PL = PrefillPlan<DK>;
    constexpr int RL = SP::RL;
    constexpr int RPC = SP::RPC;
    constexpr int NT = SP::THREADS;
    constexpr int CT = PL::CT;
    const int b = blockIdx.z, h = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = lane / SP::P, pp = lane % SP::P;
    const int row0 = blockIdx.x * RPC;

    // lane gather, then the sequence's bounds (each checked like the oracle: index first)
    const int slot = p.indices[b];
    const bool reporter = p.err != nullptr && tid == 0 && blockIdx.x == 0 && h == 0;  // once per sequence
    if (slot < 0 || slot >= p.num_slots) {
        if (slot != -1 && reporter) atomicOr(p.err, GDN_ERRBIT_INDEX);
        return;
    }
    const int lo = cu_seqlens[b], hi = cu_seqlens[b + 1];
    if (lo < 0 || hi < lo || hi > n_tokens) {
        if (reporter) atomicOr(p.err, GDN_ERRBIT_SEQLEN);
        return;
    }
    const int n = hi - lo;
    if (n == 0) return;
    const bool fresh = has_init != nullptr && has_init[b] == 0;

    TokenPrologue<DK, InT, RPC, NT> pro;
    RecurrentParams c = p;  // q..b, T: the chunk the prologue works on; o, pool_out: the running chunk
    c.cache = nullptr;
    c.steps = nullptr;
    chunk_inputs<DK, InT>(c, p, lo, min(CT, n));
    pro.prefetch(c, 0, h, row0, tid);

    // initial state, in the lane's register-slot order (LaneRows); zero for a fresh sequence
    const LaneRows<DK> lr(warp, rg, pp);
    float2 S[RL][4];
    {
        uint4 raw[RL][SL::NC];
        const StT* src = static_cast<const StT*>(p.pool_in) + (((int64_t)slot * p.HV + h) * p.DV + row0) * DK + 8 * pp;
#pragma unroll
        for (int s = 0; s < RL; ++s) {
#pragma unroll
            for (int cc = 0; cc < SL::NC; ++cc) raw[s][cc] = make_uint4(0, 0, 0, 0);
            if (!fresh && row0 + lr.row[s] < p.DV) SL::load_global(src + lr.row[s] * DK, raw[s]);
        }
#pragma unroll
        for (int s = 0; s < RL; ++s) SL::unpack(raw[s], S[s]);
    }

    // two buffers of q [CT][DK], k [CT][DK], v [CT][RPC], g, beta, kh.qh [CT]
    extern __shared__ __align__(16) float prefill_smem[];
    constexpr int V_OFF = 2 * CT * DK, G_OFF = V_OFF + CT * RPC;
    {
        float* bf = prefill_smem;
        pro.finish(c, 0, h, row0, tid, c.T, bf, bf + CT * DK, bf + V_OFF, bf + G_OFF, bf + G_OFF + CT, bf + G_OFF + 2 * CT);
    }
    __syncthreads();
    int cur = 0;
    for (int c0 = 0; c0 < n; c0 += CT) {
        const int len = min(CT, n - c0);
        const bool more = c0 + CT < n;
        chunk_outputs(c, p, (int64_t)lo + c0, !more);
        if (more) {
            chunk_inputs<DK, InT>(c, p, (int64_t)lo + c0 + CT, min(CT, n - c0 - CT));
            pro.prefetch(c, 0, h, row0, tid);  // in flight while this chunk runs
        }
        {
            const float* bf = prefill_smem + cur * PL::BUF_FLOATS;
            run_tokens<DK, StT>(c, S, lr, 0, h, row0, slot, len, pp, bf, bf + CT * DK, bf + V_OFF, RPC, bf + G_OFF,
                                bf + G_OFF + CT, bf + G_OFF + 2 * CT);
        }
        if (more) {
            float* bf = prefill_smem + (cur ^ 1) * PL::BUF_FLOATS;  // its readers finished before the last barrier
            pro.finish(c, 0, h, row0, tid, c.T, bf, bf + CT * DK, bf + V_OFF, bf + G_OFF, bf + G_OFF + CT,
                       bf + G_OFF + 2 * CT);
        }
        __syncthreads();
        cur ^= 1;
    }
}

template <typename InT, typename StT, int DK>
cudaError_t launch_prefill_dk(const RecurrentParams& p, const int32_t* cu_seqlens, const int32_t* has_init, int B,
                              int n_tokens, cudaStream_t s) {
    using SP = Split<DK>;
    static_assert(PrefillPlan<DK>::SMEM_BYTES <= 48 * 1024, "prefill buffers fit the default shared memory");
    const dim3 grid((p.DV + SP::RPC - 1) / SP::RPC, p.HV, B);
    gdn_prefill_kernel<DK, InT, StT><<<grid, SP::THREADS, PrefillPlan<DK>::SMEM_BYTES, s>>>(p, cu_seqlens, has_init,
                                                                                            n_tokens);
    return cudaGetLastError();
}

template <typename InT, typename StT>
cudaError_t launch_prefill_t(const RecurrentParams& p, const int32_t* cu, const int32_t* init, int B, int N, int DK,
                             cudaStream_t s) {
    switch (DK) {
    case 16: return launch_prefill_dk<InT, StT, 16>(p, cu, init, B, N, s);
    case 32: return launch_prefill_dk<InT, StT, 32>(p, cu, init, B, N, s);
    case 64: return launch_prefill_dk<InT, StT, 64>(p, cu, init, B, N, s);
    case 128: return launch_prefill_dk<InT, StT, 128>(p, cu, init, B, N, s);
    case 256: return launch_prefill_dk<InT, StT, 256>(p, cu, init, B, N, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_prefill(const RecurrentParams& p, const int32_t* cu_seqlens, const int32_t* has_init, int B,
                           int n_tokens, int DK, bool qkv_bf16, bool state_bf16, cudaStream_t s) {
#ifndef GDN_PREFILL_TOKEN_LOOP  // a comparison build keeps every DK on the token loop
    if (prefill_chunked_eligible(DK))
        return launch_prefill_chunked(p, cu_seqlens, has_init, B, n_tokens, DK, qkv_bf16, state_bf16, s);
#endif
    if (state_bf16)
        return qkv_bf16 ? launch_prefill_t<__nv_bfloat16, __nv_bfloat16>(p, cu_seqlens, has_init, B, n_tokens, DK, s)
                        : launch_prefill_t<float, __nv_bfloat16>(p, cu_seqlens, has_init, B, n_tokens, DK, s);
    return qkv_bf16 ? launch_prefill_t<__nv_bfloat16, float>(p, cu_seqlens, has_init, B, n_tokens, DK, s)
                    : launch_prefill_t<float, float>(p, cu_seqlens, has_init, B, n_tokens, DK, s);
}

}  // namespace gdn
