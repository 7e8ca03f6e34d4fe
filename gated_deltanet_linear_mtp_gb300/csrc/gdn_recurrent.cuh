// gdn_recurrent.cuh -- the decode / MTP-verify kernel of the gated delta rule (sm_103a).
//
// One CTA per (lane, value head, block of RPC state rows); the rows stay in registers for all T tokens
// (see gdn_common.cuh for the lane layout and the per-token update).  Several CTAs share an SM (72
// registers a thread: 7 CTAs of 128 threads), so one CTA's prologue loads overlap the others' token loops
// and stores; a persistent variant that staged the next items' state and q/k/v with bulk (TMA) copies held
// fewer warps per SM and measured slower on the verify workloads.
//
// Bytes.  The pool state is read once (16-byte loads that do not allocate in L1); each intermediate state
// (verify) is written once with streaming 16-byte stores; decode writes the final state back in place.
// q, k, v, a, b and the per-token scalars go through shared memory in a prologue.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Shared-memory floats of the kernel: q, k (T x DK each), v (T x RPC), g, beta, kh.qh (T each).
__host__ __device__ inline size_t general_smem_floats(int DK, int RPC, int T) {
    return (size_t)2 * T * DK + (size_t)T * RPC + 3 * (size_t)T;
}

template <int DK, typename InT, typename StT>
__global__ void __launch_bounds__(Split<DK>::THREADS, Split<DK>::MIN_CTAS_PER_SM)
    gdn_recurrent_kernel(const RecurrentParams p) {
    using SP = Split<DK>;
    using SL = Slice8<StT>;
    constexpr int RL = SP::RL;
    constexpr int RPC = SP::RPC;
    constexpr int NT = SP::THREADS;

    const int b = blockIdx.z;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = lane / SP::P, pp = lane % SP::P;
    const int T = p.T;

    // Loads that do not depend on the pool slot are issued together with the slot's own load: q and k of
    // the warp's first kPrefetchTokens tokens, v of the first kPrefetchV (token, row) pairs of this thread,
    // a, b, A_log, dt_bias.  Then only the state load waits for the slot.
    constexpr int QPL = (DK + 31) / 32;
    constexpr int kPrefetchTokens = 2;
    constexpr int kPrefetchV = 2;
    const int hk = h / (p.HV / p.HK);
    const int row0 = blockIdx.x * RPC;
    const int slot = p.indices[b];
    float qv[kPrefetchTokens][QPL], kv[kPrefetchTokens][QPL];
#pragma unroll
    for (int u = 0; u < kPrefetchTokens; ++u) {
        const int t = warp + u * (SP::WARPS);
        const int64_t off = (((int64_t)b * T + t) * p.HK + hk) * DK;
#pragma unroll
        for (int i = 0; i < QPL; ++i) {
            const int e = lane + 32 * i;
            const bool ok = t < T && e < DK;
            qv[u][i] = ok ? to_f32(static_cast<const InT*>(p.q)[off + e]) : 0.f;
            kv[u][i] = ok ? to_f32(static_cast<const InT*>(p.k)[off + e]) : 0.f;
        }
    }
    const InT* vp = static_cast<const InT*>(p.v);
    auto v_at = [&](int i) -> float {  // v of (token, row) pair i of this CTA, 0 beyond DV
        const int t = i / RPC, r = i - t * RPC;
        const int rr = row0 + r;
        return rr < p.DV ? to_f32(vp[(((int64_t)b * T + t) * p.HV + h) * p.DV + rr]) : 0.f;
    };
    float vpre[kPrefetchV];
#pragma unroll
    for (int u = 0; u < kPrefetchV; ++u) {
        const int i = tid + u * NT;
        vpre[u] = i < T * RPC ? v_at(i) : 0.f;
    }
    float a_raw = 0.f, b_raw = 0.f, A_h = 0.f, dt_h = 0.f;
    if (tid < T) {
        const int64_t ab = ((int64_t)b * T + tid) * p.HV + h;
        a_raw = to_f32(static_cast<const InT*>(p.a)[ab]);
        b_raw = to_f32(static_cast<const InT*>(p.b)[ab]);
        A_h = p.A_log[h];
        dt_h = p.dt_bias[h];
    }

    // lane gather: -1 = padded lane (skipped, nothing written); other out-of-range indices are recorded in
    // the error word and skipped.
    if (slot < 0 || slot >= p.num_slots) {
        if (slot != -1 && p.err != nullptr && tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(p.err, GDN_ERRBIT_INDEX);
        return;
    }
    const int64_t head_row0 = ((int64_t)slot * p.HV + h) * p.DV;

    // state load
    uint4 raw[RL][SL::NC];
#pragma unroll
    for (int i = 0; i < RL; ++i) {
        const int row = row0 + SP::row(warp, rg, i);
        if (row < p.DV) {
            SL::load_global(static_cast<const StT*>(p.pool_in) + (head_row0 + row) * DK + 8 * pp, raw[i]);
        } else {
#pragma unroll
            for (int c = 0; c < SL::NC; ++c) raw[i][c] = make_uint4(0, 0, 0, 0);
        }
    }

    // token prologue -> shared memory
    extern __shared__ float smem[];
    float* qs = smem;          // [T][DK] normalised q
    float* ks = qs + T * DK;   // [T][DK] normalised k
    float* vs = ks + T * DK;   // [T][RPC] v of this CTA's rows
    float* gs = vs + T * RPC;  // [T] decay g
    float* bs = gs + T;        // [T] beta
    float* kqs = bs + T;       // [T] kh . qh
    for (int t = warp, u = 0; t < T; t += SP::WARPS, ++u) {
        float q_[QPL], k_[QPL];
        if (u < kPrefetchTokens) {
#pragma unroll
            for (int i = 0; i < QPL; ++i) {
                q_[i] = u == 0 ? qv[0][i] : qv[kPrefetchTokens - 1][i];
                k_[i] = u == 0 ? kv[0][i] : kv[kPrefetchTokens - 1][i];
            }
        } else {
            const int64_t off = (((int64_t)b * T + t) * p.HK + hk) * DK;
#pragma unroll
            for (int i = 0; i < QPL; ++i) {
                const int e = lane + 32 * i;
                q_[i] = e < DK ? to_f32(static_cast<const InT*>(p.q)[off + e]) : 0.f;
                k_[i] = e < DK ? to_f32(static_cast<const InT*>(p.k)[off + e]) : 0.f;
            }
        }
        float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
        for (int i = 0; i < QPL; ++i) {
            sq = fmaf(q_[i], q_[i], sq);
            sk = fmaf(k_[i], k_[i], sk);
            sqk = fmaf(q_[i], k_[i], sqk);
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, m);
            sk += __shfl_xor_sync(0xffffffffu, sk, m);
            sqk += __shfl_xor_sync(0xffffffffu, sqk, m);
        }
        const float rq = 1.f / sqrtf(sq + p.l2_eps);
        const float rk = 1.f / sqrtf(sk + p.l2_eps);
#pragma unroll
        for (int i = 0; i < QPL; ++i) {
            const int e = lane + 32 * i;
            if (e < DK) {
                qs[t * DK + e] = q_[i] * rq;
                ks[t * DK + e] = k_[i] * rk;
            }
        }
        if (lane == 0) kqs[t] = sqk * rq * rk;
    }
    if (tid < T) {
        gs[tid] = gate(A_h, a_raw, dt_h);
        bs[tid] = sigmoid(b_raw);
    }
#pragma unroll
    for (int u = 0; u < kPrefetchV; ++u) {
        const int i = tid + u * NT;
        if (i < T * RPC) vs[i] = vpre[u];
    }
    for (int i = tid + kPrefetchV * NT; i < T * RPC; i += NT) vs[i] = v_at(i);
    __syncthreads();

    float2 S[RL][4];
#pragma unroll
    for (int i = 0; i < RL; ++i) SL::unpack(raw[i], S[i]);

    StT* cache = static_cast<StT*>(p.cache);
    const int own = SP::own_slot(pp);
    const int own_row = row0 + SP::row(warp, rg, own);
    const bool writes_o = pp == SP::owner_p(own) && own_row < p.DV;
    for (int t = 0; t < T; ++t) {
        const float orow =
            token_update<DK, float>(S, ks + t * DK, qs + t * DK, gs[t], bs[t], vs + t * RPC, warp, rg, pp, kqs[t]);
        if (cache != nullptr) {
            StT* dst = cache + ((((int64_t)b * T + t) * p.HV + h) * p.DV + row0) * DK + 8 * pp;
#pragma unroll
            for (int i = 0; i < RL; ++i) {
                const int r = SP::row(warp, rg, i);
                if (row0 + r < p.DV) SL::template store_global<true>(dst + (int64_t)r * DK, S[i]);
            }
        }
        if (writes_o) {
            const int64_t oi = (((int64_t)b * T + t) * p.HV + h) * p.DV + own_row;
            const float ov = p.scale * orow;
            if (p.out_bf16)
                static_cast<__nv_bfloat16*>(p.o)[oi] = __float2bfloat16_rn(ov);
            else
                static_cast<float*>(p.o)[oi] = ov;
        }
    }

    // decode write-back, in place
    if (p.pool_out != nullptr) {
        StT* dst = static_cast<StT*>(p.pool_out) + (head_row0 + row0) * DK + 8 * pp;
#pragma unroll
        for (int i = 0; i < RL; ++i) {
            const int r = SP::row(warp, rg, i);
            if (row0 + r < p.DV) SL::template store_global<false>(dst + (int64_t)r * DK, S[i]);
        }
    }
}

}  // namespace gdn
