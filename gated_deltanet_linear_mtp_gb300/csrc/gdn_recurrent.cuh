// gdn_recurrent.cuh -- the decode / MTP-verify / replay-commit kernels of the gated delta rule (sm_103a).
//
// Both kernels give one CTA of 4 warps a (lane, value head) pair and run the same token loop over blocks of
// RPC = Split<DK>::RPC state rows held in fp32 registers (gdn_common.cuh: lane layout, per-token update).
//
//   gdn_recurrent_kernel         one block of rows per CTA; the state comes straight from global memory
//                                with 16-byte loads into registers.  Many CTAs per SM overlap one CTA's
//                                prologue with the others' token loops.
//   gdn_recurrent_staged_kernel  NSUB consecutive blocks per CTA (16 or 32 KiB of state); the CTA's rows are bulk-copied
//                                (TMA) into shared memory at once, one copy and one mbarrier per block, so
//                                the bytes in flight per SM are not bounded by registers; the token
//                                prologue is formed once for all the blocks.  Used where a CTA has little
//                                work per state byte (few tokens), where the direct kernel is latency-bound.
//
// Bytes.  The pool state is read once; each intermediate state (verify) is written once with streaming
// 16-byte stores; decode and replay commit write the final state back in place.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Token prologue of a CTA covering ROWS consecutive state rows [row0, row0 + ROWS) of one (lane, head):
// normalised q and k (shared memory, columns at Split::kq_pos), v of the rows, g, beta and kh.qh per token.
// LPT = DK/8 lanes per token each own columns [8 tj, 8 tj + 8) of q and k: one 16-byte load per operand
// (two for fp32 inputs); a warp covers TPW tokens per pass.  prefetch() issues the loads that do not
// depend on the pool slot, so that they overlap the slot's own load; finish() writes shared memory.
template <int DK, typename InT, int ROWS, int NT>
struct TokenPrologue {
    using QK = Slice8<InT>;
    static constexpr int LPT = DK / 8;
    static constexpr int TPW = 32 / LPT;
    static constexpr int TPASS = (NT / 32) * TPW;
    static constexpr int VCH = 16 / sizeof(InT);  // v elements per 16-byte chunk
    static constexpr int VCPT = ROWS / VCH;       // v chunks per token
    static_assert(ROWS % VCH == 0, "v chunks tile the rows");

    __host__ __device__ static size_t smem_floats(int T) { return (size_t)2 * T * DK + (size_t)T * ROWS + 3 * (size_t)T; }

    uint4 qraw[QK::NC], kraw[QK::NC], vpre;
    InT a_raw, b_raw;  // converted in finish(): a conversion here would wait for the load
    float A_h, dt_h;
    int t0, tj, hk;

    __device__ __forceinline__ void prefetch(const RecurrentParams& p, int b, int h, int row0, int tid) {
        const int warp = tid >> 5, lane = tid & 31;
        const int T = p.T;
        tj = lane % LPT;
        t0 = warp * TPW + lane / LPT;
        hk = h / (p.HV / p.HK);
        a_raw = b_raw = InT(0.f);
#pragma unroll
        for (int c = 0; c < QK::NC; ++c) qraw[c] = kraw[c] = make_uint4(0, 0, 0, 0);
        if (t0 < T) {
            const int64_t off = (((int64_t)b * T + t0) * p.HK + hk) * DK + 8 * tj;
            QK::load_global(static_cast<const InT*>(p.q) + off, qraw);
            QK::load_global(static_cast<const InT*>(p.k) + off, kraw);
            if (tj == 0) {
                const int64_t ab = ((int64_t)b * T + t0) * p.HV + h;
                a_raw = static_cast<const InT*>(p.a)[ab];
                b_raw = static_cast<const InT*>(p.b)[ab];
            }
        }
        A_h = p.A_log[h];
        dt_h = p.dt_bias[h];
        vpre = make_uint4(0, 0, 0, 0);
        if (p.v_vec && tid < T * VCPT) {
            const int t = tid / VCPT, c = tid - t * VCPT;
            if (row0 + c * VCH < p.DV)
                vpre = ld_state16(static_cast<const InT*>(p.v) + (((int64_t)b * T + t) * p.HV + h) * p.DV + row0 + c * VCH);
        }
    }

    // qs, ks: [T][DK]; vs: [T][ROWS]; gs, bs, kqs: [T].  No barrier inside: the caller syncs.
    __device__ __forceinline__ void finish(const RecurrentParams& p, int b, int h, int row0, int tid, int steps,
                                           float* qs, float* ks, float* vs, float* gs, float* bs, float* kqs) {
        const int T = p.T;
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
                        a_raw = static_cast<const InT*>(p.a)[ab];
                        b_raw = static_cast<const InT*>(p.b)[ab];
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
                *reinterpret_cast<float4*>(qd + DK / 2) =
                    make_float4(q2[2].x * rq, q2[2].y * rq, q2[3].x * rq, q2[3].y * rq);
                *reinterpret_cast<float4*>(kd) = make_float4(k2[0].x * rk, k2[0].y * rk, k2[1].x * rk, k2[1].y * rk);
                *reinterpret_cast<float4*>(kd + DK / 2) =
                    make_float4(k2[2].x * rk, k2[2].y * rk, k2[3].x * rk, k2[3].y * rk);
                if (tj == 0) {
                    kqs[t] = sqk * rq * rk;
                    gs[t] = gate(A_h, to_f32(a_raw), dt_h);
                    bs[t] = sigmoid(to_f32(b_raw));
                }
            }
        }
        const InT* vp = static_cast<const InT*>(p.v);
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
                for (int e = 0; e < VCH; ++e) vs[t * ROWS + c * VCH + e] = f[e];
            }
        } else {
            for (int i = tid; i < steps * ROWS; i += NT) {
                const int t = i / ROWS, r = i - t * ROWS;
                const int rr = row0 + r;
                vs[i] = rr < p.DV ? to_f32(vp[(((int64_t)b * T + t) * p.HV + h) * p.DV + rr]) : 0.f;
            }
        }
    }
};

// The token loop of one block of RPC rows starting at row r0 (rows r0 + lr.row[s] of the (lane, head)):
// S holds the block's state in registers; vs_blk points at v of token 0 for the block's first row, with a
// token stride of vs_stride floats.  Stores the intermediate states, the outputs and the write-back that
// the call asks for.
// With the fused gated norm (osm != nullptr) the stored o of every row also goes to osm[t][row - cta_row0], rows of
// the CTA in a stride of osm_rows.
template <int DK, typename StT>
__device__ __forceinline__ void run_tokens(const RecurrentParams& p, float2 (&S)[Split<DK>::RL][4],
                                           const LaneRows<DK>& lr, int b, int h, int r0, int slot, int steps, int pp,
                                           const float* qs, const float* ks, const float* vs_blk, int vs_stride,
                                           const float* gs, const float* bs, const float* kqs, float* osm = nullptr,
                                           int osm_rows = 0, int cta_row0 = 0) {
    using SP = Split<DK>;
    using SL = Slice8<StT>;
    constexpr int RL = SP::RL;
    const int T = p.T;
    unsigned live = 0;  // bit s: register slot s holds a row < DV
#pragma unroll
    for (int s = 0; s < RL; ++s) live |= (r0 + lr.row[s] < p.DV ? 1u : 0u) << s;
    const int64_t tok_state = (int64_t)p.HV * p.DV * DK;  // elements between two tokens' states of a lane
    const int64_t tok_out = (int64_t)p.HV * p.DV;
    StT* cache_t = p.cache == nullptr
                       ? nullptr
                       : static_cast<StT*>(p.cache) + (((int64_t)b * T * p.HV + h) * p.DV + r0) * DK + 8 * pp;
    const int64_t o0 = ((int64_t)b * T * p.HV + h) * p.DV + r0 + lr.own_row;
    const bool writes_o = p.o != nullptr && pp == SP::owner_p(lr.code) && r0 + lr.own_row < p.DV;
    for (int t = 0; t < steps; ++t) {
        const float orow = token_update<DK>(S, ks + t * DK, qs + t * DK, gs[t], bs[t],
                                            vs_blk[t * vs_stride + lr.own_row], kqs[t], pp, lr);
        if (cache_t != nullptr) {
#pragma unroll
            for (int s = 0; s < RL; ++s)
                if (live & (1u << s)) SL::template store_global<true>(cache_t + lr.row[s] * DK, S[s]);
            cache_t += tok_state;
        }
        if (writes_o) {
            const float ov = p.scale * orow;
            float stored = ov;
            if (p.out_bf16) {
                const __nv_bfloat16 ob = __float2bfloat16_rn(ov);
                static_cast<__nv_bfloat16*>(p.o)[o0 + t * tok_out] = ob;
                stored = __bfloat162float(ob);
            } else {
                static_cast<float*>(p.o)[o0 + t * tok_out] = ov;
            }
            if (osm != nullptr) osm[t * osm_rows + (r0 - cta_row0) + lr.own_row] = stored;
        }
    }
    // decode / replay-commit write-back, in place
    if (p.pool_out != nullptr) {
        StT* dst = static_cast<StT*>(p.pool_out) + ((((int64_t)slot * p.HV + h) * p.DV) + r0) * DK + 8 * pp;
#pragma unroll
        for (int s = 0; s < RL; ++s)
            if (live & (1u << s)) SL::template store_global<false>(dst + lr.row[s] * DK, S[s]);
    }
}

// Lane gather and token count.  Returns false (the CTA has nothing to do) for a padded lane (-1), an
// out-of-range index (error bit), or a replay-commit length of 0 or outside 0..T (error bit).
__device__ __forceinline__ bool lane_work(const RecurrentParams& p, int slot, int steps, int h, int tid) {
    const bool reporter = p.err != nullptr && tid == 0 && blockIdx.x == 0 && h == 0;  // once per lane
    if (slot < 0 || slot >= p.num_slots) {
        if (slot != -1 && reporter) atomicOr(p.err, GDN_ERRBIT_INDEX);
        return false;
    }
    if (steps < 0 || steps > p.T) {
        if (reporter) atomicOr(p.err, GDN_ERRBIT_ACCEPT_LEN);
        return false;
    }
    return steps > 0;
}

// ---- the fused gated norm of the outputs --------------------------------------------------------------------
// y = o / sqrt(mean over the head's DV rows of o^2 + eps) * w * silu(z) per (token, head), o as stored.  The CTAs
// of one (lane, head) run as one thread-block cluster (grid.x of them, at most 8).  Every CTA shares the lane and the
// head, so all of them take the same early exit or none.
//   norm_begin     (after the lane check) arrives on the cluster barrier's first phase (this CTA has started: its
//                  shared memory may be written by the others) and gathers the CTA's z rows into shared memory with
//                  16-byte cp.async copies, which overlap the state load and the token loop;
//   norm_epilogue  sums o^2 over the CTA's rows per token and stores the sums into every CTA's slot for this rank
//                  (distributed shared memory), one barrier phase, then every CTA adds the ranks' sums in rank order
//                  (all see the same value) and writes y for its rows.  No CTA touches another's shared memory after
//                  that phase, so each may leave when it is done.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctas() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(float* local, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

constexpr int kNormMaxCluster = 8;  // CTAs of one head in a cluster at most (the portable cluster size)

// The norm's shared memory after the kernel's own `base` bytes, for T tokens of `rows` rows:
//   zs    [T][rows] z as given (bf16 or fp32; 4 bytes an element reserved), 16-byte aligned
//   os    [T][rows] the stored o of the rows, fp32
//   part  [kNormMaxCluster][GDN_MAX_T] every rank's sums of o^2 per token
//   inv   [GDN_MAX_T] 1 / rms of the head per token
struct NormSmem {
    __host__ __device__ static size_t zs(size_t base) { return (base + 15) & ~(size_t)15; }
    __host__ __device__ static size_t os(size_t base, int T, int rows) { return zs(base) + sizeof(float) * T * rows; }
    __host__ __device__ static size_t part(size_t base, int T, int rows) {
        return os(base, T, rows) + sizeof(float) * T * rows;
    }
    __host__ __device__ static size_t end(size_t base, int T, int rows) {
        return part(base, T, rows) + sizeof(float) * (kNormMaxCluster + 1) * GDN_MAX_T;
    }
};

// zs: the CTA's rows row0 .. row0 + rows - 1 of z for T tokens (chunks of rows past DV are not copied)
__device__ __forceinline__ void norm_begin(const RecurrentParams& p, unsigned char* zs, int rows, int row0, int b,
                                           int h, int T, int tid, int nt) {
    cluster_arrive_relaxed();
    if (!p.nz_vec) return;
    const int zb = p.nz_bf16 ? 2 : 4;
    const int zch = 16 / zb;  // elements per chunk; DV % 8 == 0 puts every chunk wholly inside or past DV
    const int cpt = rows / zch;
    const unsigned char* z = static_cast<const unsigned char*>(p.nz);
    for (int i = tid; i < T * cpt; i += nt) {
        const int t = i / cpt, c = i - t * cpt, row = row0 + c * zch;
        if (row < p.DV)
            cp_async16(zs + (size_t)(t * rows + c * zch) * zb,
                       z + ((((int64_t)b * T + t) * p.HV + h) * p.DV + row) * zb);
    }
}

// os: [T][rows] stored o of the CTA's rows row0 .. row0 + rows - 1; zs as norm_begin left it
template <int NT>
__device__ __forceinline__ void norm_epilogue(const RecurrentParams& p, const unsigned char* zs, const float* os,
                                              float* part, int rows, int row0, int b, int h, int T, int tid) {
    float* inv = part + kNormMaxCluster * GDN_MAX_T;
    const int warp = tid >> 5, lane = tid & 31;
    cp_async_commit_wait_all();
    __syncthreads();      // every row's o and z are in place
    cluster_wait_acquire();  // every CTA of the cluster has started
    const uint32_t n = cluster_ctas(), me = cluster_rank();
    for (int t = warp; t < T; t += NT / 32) {
        float sq = 0.f;
        for (int r = lane; r < rows; r += 32)
            if (row0 + r < p.DV) sq = fmaf(os[t * rows + r], os[t * rows + r], sq);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, m);
        if ((uint32_t)lane < n) st_cluster_f32(part + me * GDN_MAX_T + t, (uint32_t)lane, sq);
    }
    cluster_arrive_release();
    cluster_wait_acquire();  // every rank's sums are in every CTA's part
    if (tid < T) {
        float tot = 0.f;
        for (uint32_t r = 0; r < n; ++r) tot += part[r * GDN_MAX_T + tid];
        inv[tid] = 1.f / sqrtf(tot / (float)p.DV + p.neps);
    }
    __syncthreads();
    const int64_t tok_out = (int64_t)p.HV * p.DV;
    for (int i = tid; i < T * rows; i += NT) {
        const int t = i / rows, r = i - t * rows, row = row0 + r;
        if (row >= p.DV) continue;
        const int64_t off = ((int64_t)b * T + t) * tok_out + (int64_t)h * p.DV + row;
        float zt;
        if (p.nz_vec)
            zt = p.nz_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(zs)[i])
                           : reinterpret_cast<const float*>(zs)[i];
        else
            zt = p.nz_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.nz)[off])
                           : static_cast<const float*>(p.nz)[off];
        const float y = os[i] * inv[t] * p.nw[row] * (zt / (1.f + expf(-zt)));
        if (p.out_bf16)
            static_cast<__nv_bfloat16*>(p.ny)[off] = __float2bfloat16_rn(y);
        else
            static_cast<float*>(p.ny)[off] = y;
    }
}

template <int DK>
__host__ __device__ inline size_t direct_smem_bytes(int T) {
    return sizeof(float) * TokenPrologue<DK, float, Split<DK>::RPC, Split<DK>::THREADS>::smem_floats(T);
}

// (with the fused norm, one CTA per SM less of register budget: its epilogue's values would spill otherwise)
template <int DK, typename InT, typename StT, bool kNorm = false>
__global__ void __launch_bounds__(Split<DK>::THREADS, Split<DK>::MIN_CTAS_PER_SM - (kNorm ? 1 : 0))
    gdn_recurrent_kernel(const RecurrentParams p) {
    using SP = Split<DK>;
    using SL = Slice8<StT>;
    constexpr int RL = SP::RL;
    constexpr int RPC = SP::RPC;
    constexpr int NT = SP::THREADS;
    const int b = blockIdx.z, h = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = lane / SP::P, pp = lane % SP::P;
    const int T = p.T;
    const int row0 = blockIdx.x * RPC;

    // Loads that do not depend on the pool slot go out with the slot's own load; then only the state load
    // waits for the slot.
    const int slot = p.indices[b];
    const int steps = p.steps != nullptr ? p.steps[b] : T;
    TokenPrologue<DK, InT, RPC, NT> pro;
    pro.prefetch(p, b, h, row0, tid);
    if (!lane_work(p, slot, steps, h, tid)) return;
    extern __shared__ __align__(16) float smem[];
    unsigned char* const norm_base = reinterpret_cast<unsigned char*>(smem);
    if constexpr (kNorm) norm_begin(p, norm_base + NormSmem::zs(direct_smem_bytes<DK>(T)), RPC, row0, b, h, T, tid, NT);

    // state load, in the lane's register-slot order (LaneRows)
    const LaneRows<DK> lr(warp, rg, pp);
    uint4 raw[RL][SL::NC];
    {
        const StT* src = static_cast<const StT*>(p.pool_in) + (((int64_t)slot * p.HV + h) * p.DV + row0) * DK + 8 * pp;
#pragma unroll
        for (int s = 0; s < RL; ++s) {
            if (row0 + lr.row[s] < p.DV) {
                SL::load_global(src + lr.row[s] * DK, raw[s]);
            } else {
#pragma unroll
                for (int c = 0; c < SL::NC; ++c) raw[s][c] = make_uint4(0, 0, 0, 0);
            }
        }
    }

    float* qs = smem;          // [T][DK] normalised q, columns permuted by Split::kq_pos
    float* ks = qs + T * DK;   // [T][DK] normalised k, likewise
    float* vs = ks + T * DK;   // [T][RPC] v of this CTA's rows
    float* gs = vs + T * RPC;  // [T] decay g
    float* bs = gs + T;        // [T] beta
    float* kqs = bs + T;       // [T] kh . qh
    pro.finish(p, b, h, row0, tid, steps, qs, ks, vs, gs, bs, kqs);
    __syncthreads();

    float2 S[RL][4];
#pragma unroll
    for (int s = 0; s < RL; ++s) SL::unpack(raw[s], S[s]);
    const size_t nb = direct_smem_bytes<DK>(T);
    float* osm = kNorm ? reinterpret_cast<float*>(norm_base + NormSmem::os(nb, T, RPC)) : nullptr;
    run_tokens<DK, StT>(p, S, lr, b, h, row0, slot, steps, pp, qs, ks, vs, RPC, gs, bs, kqs, osm, RPC, row0);
    if constexpr (kNorm)
        norm_epilogue<NT>(p, norm_base + NormSmem::zs(nb), osm,
                          reinterpret_cast<float*>(norm_base + NormSmem::part(nb, T, RPC)), RPC, row0, b, h, T, tid);
}

// ---- TMA-staged kernel ------------------------------------------------------------------------------------
constexpr uint32_t kMbarPollLimit = GDN_WAIT_POLLS;  // polls of one mbarrier wait before it is declared failed

template <int DK, typename StT, int KIB>
struct Staged {
    static constexpr int RPC = Split<DK>::RPC;
    static constexpr int BLOCK_BYTES = RPC * DK * (int)sizeof(StT);
    // up to KIB KiB of state per CTA, in NSUB blocks of RPC rows
    static constexpr int CAP = KIB * 1024;
    static constexpr int NSUB = BLOCK_BYTES >= CAP ? 1 : (CAP / BLOCK_BYTES > 8 ? 8 : CAP / BLOCK_BYTES);
    static constexpr int ROWS = NSUB * RPC;
    // resident CTAs the register budget aims at: 7 (70 registers, no spills) for the fp32 16 KiB stage at
    // DK = 128, which measured 6-9% faster than 6 on T = 1 decodes; 6 elsewhere
    static constexpr int MIN_CTAS = (sizeof(StT) == 4 && KIB == 16 && DK == 128) ? 7 : Split<DK>::MIN_CTAS_PER_SM;
    __host__ __device__ static uint32_t prologue_offset() { return (uint32_t)NSUB * BLOCK_BYTES; }
    __host__ __device__ static uint32_t mbar_offset(int T) {
        const uint32_t end =
            prologue_offset() +
            (uint32_t)(sizeof(float) * TokenPrologue<DK, float, ROWS, Split<DK>::THREADS>::smem_floats(T));
        return (end + 15u) & ~15u;
    }
    __host__ __device__ static uint32_t smem_bytes(int T) { return mbar_offset(T) + 8u * NSUB; }
    __host__ __device__ static uint32_t norm_offset(int T) { return (smem_bytes(T) + 15u) & ~15u; }
};

template <int DK, typename InT, typename StT, int KIB, bool kNorm = false>
__global__ void __launch_bounds__(Split<DK>::THREADS, Staged<DK, StT, KIB>::MIN_CTAS - (kNorm ? 1 : 0))
    gdn_recurrent_staged_kernel(const RecurrentParams p) {
    using SP = Split<DK>;
    using SL = Slice8<StT>;
    using ST = Staged<DK, StT, KIB>;
    constexpr int RL = SP::RL;
    constexpr int RPC = SP::RPC;
    constexpr int NT = SP::THREADS;
    constexpr int NSUB = ST::NSUB;
    constexpr int ROWS = ST::ROWS;
    const int b = blockIdx.z, h = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = lane / SP::P, pp = lane % SP::P;
    const int T = p.T;
    const int row0 = blockIdx.x * ROWS;

    const int slot = p.indices[b];
    const int steps = p.steps != nullptr ? p.steps[b] : T;
    TokenPrologue<DK, InT, ROWS, NT> pro;
    pro.prefetch(p, b, h, row0, tid);
    if (!lane_work(p, slot, steps, h, tid)) return;

    extern __shared__ __align__(16) unsigned char staged_smem[];
    const size_t nb = ST::norm_offset(T);
    if constexpr (kNorm) norm_begin(p, staged_smem + NormSmem::zs(nb), ROWS, row0, b, h, T, tid, NT);
    const uint32_t sbase = smem_u32(staged_smem);
    const uint32_t mbar0 = sbase + ST::mbar_offset(T);
    if (tid == 0) {
        for (int s = 0; s < NSUB; ++s) mbar_init(mbar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // one bulk copy per block of rows, each completing on its own mbarrier (used once: phase parity 0)
    const int64_t head_row0 = ((int64_t)slot * p.HV + h) * p.DV;
    if (tid < NSUB) {
        const int r = row0 + tid * RPC;
        const int nrows = min(RPC, p.DV - r);
        bool issue_copy = nrows > 0;
#ifdef GDN_TEST_MISSING_COPY
        // test build: block 0 of the first CTA is never copied (and never arrived on), so its wait runs out
        if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) issue_copy = false;
#endif
        if (issue_copy) {
            const uint32_t bytes = (uint32_t)nrows * DK * sizeof(StT);
            mbar_arrive_expect_tx(mbar0 + 8 * tid, bytes);
            bulk_g2s(sbase + (uint32_t)tid * ST::BLOCK_BYTES, static_cast<const StT*>(p.pool_in) + (head_row0 + r) * DK,
                     bytes, mbar0 + 8 * tid);
        }
    }

    float* qs = reinterpret_cast<float*>(staged_smem + ST::prologue_offset());
    float* ks = qs + T * DK;
    float* vs = ks + T * DK;  // [T][ROWS]
    float* gs = vs + T * ROWS;
    float* bs = gs + T;
    float* kqs = bs + T;
    pro.finish(p, b, h, row0, tid, steps, qs, ks, vs, gs, bs, kqs);
    __syncthreads();

    const LaneRows<DK> lr(warp, rg, pp);
    float* osm = kNorm ? reinterpret_cast<float*>(staged_smem + NormSmem::os(nb, T, ROWS)) : nullptr;
    bool failed = false;
    for (int sb = 0; sb < NSUB; ++sb) {
        const int r0 = row0 + sb * RPC;
        if (r0 >= p.DV) break;
        const uint32_t bar = mbar0 + 8 * sb;
        // bounded wait; the whole warp skips a block whose copy did not land (its shuffles need every lane)
        if (__any_sync(0xffffffffu, !mbar_wait_bounded(bar, 0, kMbarPollLimit))) {
            failed = true;
            mbar_wait_bounded(bar, 0, kMbarPollLimit);  // one more bounded chance for a late copy to drain
            continue;
        }
        const StT* tile = reinterpret_cast<const StT*>(staged_smem + sb * ST::BLOCK_BYTES) + 8 * pp;
        float2 S[RL][4];
#pragma unroll
        for (int s = 0; s < RL; ++s) SL::load_shared(tile + lr.row[s] * DK, S[s]);
        run_tokens<DK, StT>(p, S, lr, b, h, r0, slot, steps, pp, qs, ks, vs + sb * RPC, ROWS, gs, bs, kqs, osm, ROWS,
                            row0);
    }
    if (failed && lane == 0 && p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_TIMEOUT);
    if constexpr (kNorm)
        norm_epilogue<NT>(p, staged_smem + NormSmem::zs(nb), osm,
                          reinterpret_cast<float*>(staged_smem + NormSmem::part(nb, T, ROWS)), ROWS, row0, b, h, T, tid);
}

}  // namespace gdn
