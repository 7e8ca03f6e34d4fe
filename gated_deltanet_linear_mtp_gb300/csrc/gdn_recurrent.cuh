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

    // Token prologue layout: LPT = DK/8 lanes per token, each lane owning columns [8 tj, 8 tj + 8) of the
    // token's q and k, so one 16-byte load per operand (two for fp32); a warp covers TPW tokens per pass.
    using QK = Slice8<InT>;
    constexpr int LPT = DK / 8;
    constexpr int TPW = 32 / LPT;
    constexpr int TPASS = SP::WARPS * TPW;
    constexpr int VCH = 16 / sizeof(InT);  // v elements per 16-byte chunk
    const int tg = lane / LPT, tj = lane % LPT;
    const int hk = h / (p.HV / p.HK);
    const int row0 = blockIdx.x * RPC;

    // Loads that do not depend on the pool slot are issued together with the slot's own load: q, k, a, b
    // of the first pass's tokens, the first 16-byte chunk of v of this thread, A_log and dt_bias.  Then
    // only the state load waits for the slot.
    const int slot = p.indices[b];
    const int steps = p.steps != nullptr ? p.steps[b] : T;
    const int t0 = warp * TPW + tg;
    uint4 qraw[QK::NC], kraw[QK::NC];
    float a_raw = 0.f, b_raw = 0.f;
    if (t0 < T) {
        const int64_t off = (((int64_t)b * T + t0) * p.HK + hk) * DK + 8 * tj;
        QK::load_global(static_cast<const InT*>(p.q) + off, qraw);
        QK::load_global(static_cast<const InT*>(p.k) + off, kraw);
        if (tj == 0) {
            const int64_t ab = ((int64_t)b * T + t0) * p.HV + h;
            a_raw = to_f32(static_cast<const InT*>(p.a)[ab]);
            b_raw = to_f32(static_cast<const InT*>(p.b)[ab]);
        }
    }
    const float A_h = p.A_log[h], dt_h = p.dt_bias[h];
    const InT* vp = static_cast<const InT*>(p.v);
    constexpr int VCPT = RPC / VCH;  // v chunks per token
    uint4 vpre = make_uint4(0, 0, 0, 0);
    if (p.v_vec && tid < T * VCPT) {
        const int t = tid / VCPT, c = tid - t * VCPT;
        if (row0 + c * VCH < p.DV)
            vpre = ld_state16(vp + (((int64_t)b * T + t) * p.HV + h) * p.DV + row0 + c * VCH);
    }

    // lane gather: -1 = padded lane (skipped, nothing written); other out-of-range indices are recorded in
    // the error word and skipped.
    if (slot < 0 || slot >= p.num_slots) {
        if (slot != -1 && p.err != nullptr && tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(p.err, GDN_ERRBIT_INDEX);
        return;
    }
    // replay commit: steps[b] tokens; 0 = nothing to commit; outside 0..T = recorded and skipped
    if (steps < 0 || steps > T) {
        if (p.err != nullptr && tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(p.err, GDN_ERRBIT_ACCEPT_LEN);
        return;
    }
    if (steps == 0) return;
    const int64_t head_row0 = ((int64_t)slot * p.HV + h) * p.DV;

    // state load, in the lane's register-slot order (LaneRows)
    const LaneRows<DK> lr(warp, rg, pp);
    unsigned live = 0;  // bit s: register slot s holds a row < DV
#pragma unroll
    for (int s = 0; s < RL; ++s) live |= (row0 + lr.row[s] < p.DV ? 1u : 0u) << s;
    uint4 raw[RL][SL::NC];
    {
        const StT* src = static_cast<const StT*>(p.pool_in) + (head_row0 + row0) * DK + 8 * pp;
#pragma unroll
        for (int s = 0; s < RL; ++s) {
            if (live & (1u << s)) {
                SL::load_global(src + lr.row[s] * DK, raw[s]);
            } else {
#pragma unroll
                for (int c = 0; c < SL::NC; ++c) raw[s][c] = make_uint4(0, 0, 0, 0);
            }
        }
    }

    // token prologue -> shared memory
    extern __shared__ float smem[];
    float* qs = smem;          // [T][DK] normalised q, columns permuted by Split::kq_pos
    float* ks = qs + T * DK;   // [T][DK] normalised k, likewise
    float* vs = ks + T * DK;   // [T][RPC] v of this CTA's rows
    float* gs = vs + T * RPC;  // [T] decay g
    float* bs = gs + T;        // [T] beta
    float* kqs = bs + T;       // [T] kh . qh
    for (int pass = 0; pass * TPASS < steps; ++pass) {
        const int t = t0 + pass * TPASS;
        if (pass > 0) {
#pragma unroll
            for (int c = 0; c < QK::NC; ++c) qraw[c] = kraw[c] = make_uint4(0, 0, 0, 0);
            if (t < steps) {
                const int64_t off = (((int64_t)b * T + t) * p.HK + hk) * DK + 8 * tj;
                QK::load_global(static_cast<const InT*>(p.q) + off, qraw);
                QK::load_global(static_cast<const InT*>(p.k) + off, kraw);
                if (tj == 0) {
                    const int64_t ab = ((int64_t)b * T + t) * p.HV + h;
                    a_raw = to_f32(static_cast<const InT*>(p.a)[ab]);
                    b_raw = to_f32(static_cast<const InT*>(p.b)[ab]);
                }
            }
        }
        float2 q2[4], k2[4];
        QK::unpack(qraw, q2);
        QK::unpack(kraw, k2);
        float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            sq = fmaf(q2[e].x, q2[e].x, fmaf(q2[e].y, q2[e].y, sq));
            sk = fmaf(k2[e].x, k2[e].x, fmaf(k2[e].y, k2[e].y, sk));
            sqk = fmaf(q2[e].x, k2[e].x, fmaf(q2[e].y, k2[e].y, sqk));
        }
#pragma unroll
        for (int m = 1; m < LPT; m <<= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, m);
            sk += __shfl_xor_sync(0xffffffffu, sk, m);
            sqk += __shfl_xor_sync(0xffffffffu, sqk, m);
        }
        if (t < steps) {
            const float rq = 1.f / sqrtf(sq + p.l2_eps);
            const float rk = 1.f / sqrtf(sk + p.l2_eps);
            // columns [8 tj, 8 tj + 4) sit at 4 tj, [8 tj + 4, 8 tj + 8) at DK/2 + 4 tj (Split::kq_pos)
            float* qd = qs + t * DK + 4 * tj;
            float* kd = ks + t * DK + 4 * tj;
            *reinterpret_cast<float4*>(qd) = make_float4(q2[0].x * rq, q2[0].y * rq, q2[1].x * rq, q2[1].y * rq);
            *reinterpret_cast<float4*>(qd + DK / 2) = make_float4(q2[2].x * rq, q2[2].y * rq, q2[3].x * rq, q2[3].y * rq);
            *reinterpret_cast<float4*>(kd) = make_float4(k2[0].x * rk, k2[0].y * rk, k2[1].x * rk, k2[1].y * rk);
            *reinterpret_cast<float4*>(kd + DK / 2) = make_float4(k2[2].x * rk, k2[2].y * rk, k2[3].x * rk, k2[3].y * rk);
            if (tj == 0) {
                kqs[t] = sqk * rq * rk;
                gs[t] = gate(A_h, a_raw, dt_h);
                bs[t] = sigmoid(b_raw);
            }
        }
    }
    if (p.v_vec) {
        for (int i = tid; i < steps * VCPT; i += NT) {
            const int t = i / VCPT, c = i - t * VCPT;
            uint4 raw_v = vpre;
            if (i != tid) {
                raw_v = make_uint4(0, 0, 0, 0);
                if (row0 + c * VCH < p.DV)
                    raw_v = ld_state16(vp + (((int64_t)b * T + t) * p.HV + h) * p.DV + row0 + c * VCH);
            }
            float f[VCH];
            Chunk<InT>::unpack(raw_v, f);
#pragma unroll
            for (int e = 0; e < VCH; ++e) vs[t * RPC + c * VCH + e] = f[e];
        }
    } else {
        for (int i = tid; i < steps * RPC; i += NT) {
            const int t = i / RPC, r = i - t * RPC;
            const int rr = row0 + r;
            vs[i] = rr < p.DV ? to_f32(vp[(((int64_t)b * T + t) * p.HV + h) * p.DV + rr]) : 0.f;
        }
    }
    __syncthreads();

    float2 S[RL][4];
#pragma unroll
    for (int i = 0; i < RL; ++i) SL::unpack(raw[i], S[i]);

    // token loop: everything per lane that does not change with the token is fixed here
    const int64_t tok_state = (int64_t)p.HV * p.DV * DK;  // elements between two tokens' states of a lane
    const int64_t tok_out = (int64_t)p.HV * p.DV;
    StT* cache_t = p.cache == nullptr ? nullptr
                                      : static_cast<StT*>(p.cache) + (((int64_t)b * T * p.HV + h) * p.DV + row0) * DK + 8 * pp;
    const int64_t o0 = ((int64_t)b * T * p.HV + h) * p.DV + row0 + lr.own_row;
    const bool writes_o = p.o != nullptr && pp == SP::owner_p(lr.code) && row0 + lr.own_row < p.DV;
    for (int t = 0; t < steps; ++t) {
        const float orow = token_update<DK>(S, ks + t * DK, qs + t * DK, gs[t], bs[t], vs[t * RPC + lr.own_row],
                                            kqs[t], pp, lr);
        if (cache_t != nullptr) {
#pragma unroll
            for (int s = 0; s < RL; ++s)
                if (live & (1u << s)) SL::template store_global<true>(cache_t + lr.row[s] * DK, S[s]);
            cache_t += tok_state;
        }
        if (writes_o) {
            const float ov = p.scale * orow;
            if (p.out_bf16)
                static_cast<__nv_bfloat16*>(p.o)[o0 + t * tok_out] = __float2bfloat16_rn(ov);
            else
                static_cast<float*>(p.o)[o0 + t * tok_out] = ov;
        }
    }

    // decode / replay-commit write-back, in place
    if (p.pool_out != nullptr) {
        StT* dst = static_cast<StT*>(p.pool_out) + (head_row0 + row0) * DK + 8 * pp;
#pragma unroll
        for (int s = 0; s < RL; ++s)
            if (live & (1u << s)) SL::template store_global<false>(dst + lr.row[s] * DK, S[s]);
    }
}

}  // namespace gdn
