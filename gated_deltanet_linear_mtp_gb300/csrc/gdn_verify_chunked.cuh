// gdn_verify_chunked.cuh -- MTP verify without intermediate states, and the replay commit, in chunked form on
// the tensor cores (tcgen05, accumulators in tensor memory); persistent CTAs stream the state tiles through a
// ring of TMA stages.
//
// When nothing needs the states S_1..S_T themselves, the recurrence can be unrolled.  Writing
// gamma_t = g_1 ... g_t, G(s,t) = g_{s+1} ... g_t (G(t,t) = 1) and delta_t = beta_t (v_t - u_t),
// S_t = g_t S_{t-1} + delta_t kh_t^T unrolls to
//     S_t = gamma_t S_0 + sum_{s<=t} G(s,t) delta_s kh_s^T,
// so for every state row
//     u_t = g_t S_{t-1} kh_t = gamma_t (S_0 kh_t) + sum_{s<t}  G(s,t) (kh_s . kh_t) delta_s
//     o_t = S_t qh_t         = gamma_t (S_0 qh_t) + sum_{s<=t} G(s,t) (kh_s . qh_t) delta_s .
// The only per-element work is the contraction P = S_0 [kh_1..kh_T qh_1..qh_T], a (128 x DK) x (DK x 2T)
// product per item.  One thread issues it as DK/16 tcgen05.mma instructions (M = 128, N = 16 or 32, bf16 in,
// fp32 accumulate in tensor memory) straight from the TMA stage, with S_0 exact in bf16 and kh, qh split into
// bf16 hi + lo parts (4T columns), which keeps about 16 significant bits of kh and qh; every thread then reads
// the P row of its own state row out of tensor memory (tcgen05.ld, lane = row).  The T x T Gram matrices
// kh.kh and kh.qh are formed with mma.sync from the same hi + lo rows, and each row's small triangular
// recurrence runs in fp32 registers, one thread per row.
//
// Three modes, for bf16 state pools, T <= 8 and DK in {64, 128, 256} (the launcher's choice):
//   verify                     outputs o only: no intermediate states, no write-back.  A stage is refilled as
//                              soon as the MMA that reads it has completed, before the row recurrence runs;
//   replay commit              the first L = steps[b] tokens, no outputs, and the state after them,
//                              S_L = gamma_L S_0 + sum_{s<L} G(s, L-1) delta_s kh_s^T, written back into the
//                              slot (kh only: 2T columns, one Gram matrix).  The rank-L update is one more
//                              tcgen05.mma: the per-row coefficients go to tensor memory (tcgen05.st, A operand),
//                              B is the kh hi / lo rows read MN-major; each thread adds gamma_L S_0 to its row
//                              of the product and writes the row over the stage, which a TMA store writes back;
//   replay commit + verify     the replay commit of an earlier call's accepted tokens, then verify of this
//                              call's tokens from the committed state as written (the rows over the stage): one
//                              read and one write of every state for a whole speculative step.
//
// Work item = 128 state rows of one (lane, value head); items are numbered row block fastest, then value
// head, then lane, and each CTA (4 warps, warp w owning rows [32w, 32w + 32)) takes a contiguous range of
// them.  One thread (PT) keeps the next state tiles in flight: one 3-D TMA tensor load per 64-column box into
// a 1024-byte aligned stage, rows past DV filled with zeros, 16-byte chunks swizzled within each 128-byte row
// (the 128-byte swizzle, which is also the K-major operand layout of tcgen05.mma and keeps the ldmatrix reads
// conflict-free).  The same thread issues the tile's MMAs.  q, k, v, a and b of the next item are loaded into
// registers while the current one is computed, and consecutive items of one key head reuse its normalised q, k
// and Gram matrices.
#pragma once

#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "gdn_common.cuh"
#include "gdn_tcgen05.cuh"

namespace gdn {

constexpr int kChunkRows = 128;  // state rows per item: 4 warps x 32 = the MMA's M
constexpr int kChunkGroupThreads = 128;  // one group of 4 warps works on one item at a time
constexpr int kChunkMaxT = 8;
constexpr int kChunkMinDK = 64;  // rows of 64 bf16 at least: whole 128-byte swizzle spans
constexpr uint32_t kChunkWaitPolls = GDN_WAIT_POLLS;
constexpr int kChunkMaxGroups = 3;
// the one-pass mode (replay commit + verify) holds both token sets: it takes at most 4 tokens in each, where three
// groups fit; with more, the two calls measured faster as separate launches of three groups each
constexpr int kFusedMaxT = 4;

// The chunked kernel's modes: verify only, replay commit only, and replay commit then verify in one pass.
enum ChunkMode { kModeVerify = 0, kModeReplay = 1, kModeReplayVerify = 2 };

// Shared-memory plan of one group, as byte offsets from its 1024-byte aligned base; the groups of a CTA sit
// one after another, then a word for the tensor-memory address.  Tr = tokens of the replay set (0 in verify
// mode), Tv = tokens of the verify set (0 in replay mode).
template <int DK, int kMode, int NS>
struct ChunkPlan {
    static_assert(DK % 64 == 0, "the chunked kernel takes whole 128-byte rows");
    // the replay modes read a stage's slot and token count at the top of an item, before that item's refill: the
    // tile (and its slot) must have been issued an item earlier, so they need two stages at least
    static_assert(kMode == kModeVerify ? NS >= 1 : NS >= 2, "stages of the chunked kernel");
    static constexpr bool kReplay = kMode != kModeVerify;
    static constexpr bool kVerify = kMode != kModeReplay;
    static constexpr int NBOX = DK / 64;                      // 64-column (128-byte) boxes per row
    static constexpr uint32_t BOX_BYTES = kChunkRows * 128;   // one box of a stage
    static constexpr uint32_t STAGE_BYTES = kChunkRows * DK * 2;
    // replay set: P columns kh hi | kh lo (2 Tr), the MMA's N a multiple of 16; B rows kh hi | kh lo | kh hi
    // (3 Tr, the write-back's K, against coefficients [c hi | c hi | c lo]) padded with zero rows to 16
    __host__ __device__ static constexpr int nr(int Tr) { return (2 * Tr + 15) / 16 * 16; }
    __host__ __device__ static constexpr int rrows(int Tr) { return kReplay ? (3 * Tr + 15) / 16 * 16 : 0; }
    // verify set: B rows kh hi | kh lo | qh hi | qh lo (4 Tv) padded to 16, also the MMA's N
    __host__ __device__ static constexpr int vrows(int Tv) { return kVerify ? (4 * Tv + 15) / 16 * 16 : 0; }
    __host__ __device__ static constexpr uint32_t br_off() { return NS * STAGE_BYTES; }
    __host__ __device__ static constexpr uint32_t bv_off(int Tr) { return br_off() + (uint32_t)rrows(Tr) * DK * 2; }
    // g, beta of the replay set (Tr each), then of the verify set (Tv each)
    __host__ __device__ static constexpr uint32_t s_off(int Tr, int Tv) {
        return bv_off(Tr) + (uint32_t)vrows(Tv) * DK * 2;
    }
    // the Gram matrices, transposed (row t holds kh_s . kh_t or kh_s . qh_t over s, padded to tp(T) floats):
    // replay kh.kh (Tr rows), then verify kh.kh and kh.qh (Tv rows each)
    __host__ __device__ static constexpr int tp(int T) { return (T + 3) & ~3; }
    __host__ __device__ static constexpr uint32_t gram_off(int Tr, int Tv) {
        return s_off(Tr, Tv) + ((8u * (Tr + Tv) + 15u) & ~15u);
    }
    // NS tile mbarriers and the MMA mbarrier, a failure flag, then per stage the pool slot (-1: nothing loaded)
    // and the token count of its item
    __host__ __device__ static constexpr uint32_t ctl_off(int Tr, int Tv) {
        return gram_off(Tr, Tv) + 4u * (uint32_t)(Tr * tp(Tr) + 2 * Tv * tp(Tv));
    }
    // verify with the gated norm: each warp's partial sums of squares, 8 tokens x 4 warps
    __host__ __device__ static constexpr uint32_t red_off(int Tr, int Tv) {
        return (ctl_off(Tr, Tv) + 8u * (NS + 1) + 8u + 8u * NS + 15u) & ~15u;
    }
    __host__ __device__ static constexpr uint32_t group_bytes(int Tr, int Tv) {
        return (red_off(Tr, Tv) + (kVerify ? 4u * 4 * kChunkMaxT : 0u) + 1023u) & ~1023u;
    }
    __host__ __device__ static constexpr uint32_t bytes(int Tr, int Tv, int G) {
        return (uint32_t)G * group_bytes(Tr, Tv) + 16u + 1024u;  // + the tensor-memory address, + alignment slack
    }
    // tokens of a set at most: kChunkMaxT, kFusedMaxT in the one-pass mode
    static constexpr int MAXT = kMode == kModeReplayVerify ? kFusedMaxT : kChunkMaxT;
    // the largest plan: MAXT tokens in each set the mode has
    __host__ __device__ static constexpr uint32_t max_bytes(int G) {
        return bytes(kReplay ? MAXT : 0, kVerify ? MAXT : 0, G);
    }
    // tensor-memory columns of one group: P; in the replay modes also the product D (DK columns, P overlaps its
    // first ones), then the coefficients, two bf16 per column
    __host__ __device__ static constexpr uint32_t a2_col() { return DK; }
    __host__ __device__ static constexpr uint32_t tmem_cols() { return kReplay ? (DK + 16 + 31) / 32 * 32 : 32; }
};

// One group's barrier (named barrier `id`, its 128 threads), and the same with an OR over a predicate.
__device__ __forceinline__ void group_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kChunkGroupThreads) : "memory");
}
__device__ __forceinline__ bool group_sync_or(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "n"(kChunkGroupThreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// d += a (16x16, row) * b (16x8, col): bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// T floats from shared memory: float4 loads when the address is 16-byte aligned by construction
template <int N, bool kVec>
__device__ __forceinline__ void load_row(const float* src, float (&dst)[N]) {
    if constexpr (kVec && N % 4 == 0) {
#pragma unroll
        for (int j = 0; j < N / 4; ++j) {
            const float4 f = reinterpret_cast<const float4*>(src)[j];
            dst[4 * j] = f.x;
            dst[4 * j + 1] = f.y;
            dst[4 * j + 2] = f.z;
            dst[4 * j + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j) dst[j] = src[j];
    }
}

// One row's T x T recurrence (T fixed at compile time, so delta stays in registers).  pr: the row of P,
// [S_0 kh hi | S_0 kh lo | S_0 qh hi | S_0 qh lo]; v: the row's v per token; KKt, KQt: the transposed Gram
// matrices, rows of TP = gram_stride(T) floats.  ost: the values stored into o (after rounding to its type).
template <int T, int NP>
__device__ __forceinline__ void row_recurrence(const RecurrentParams& p, const float (&pr)[NP], const float* v,
                                               const float* gs, const float* bs,
                                               const float* KKt, const float* KQt, bool live, int64_t o0,
                                               int64_t tok_out, float (&ost)[T]) {
    constexpr int TP = (T + 3) & ~3;
    float g[T], be[T];
    load_row<T, false>(gs, g);
    load_row<T, false>(bs, be);
    float delta[T];
    float gamma = 1.f;
#pragma unroll
    for (int t = 0; t < T; ++t) {
        float kk[TP], kq[TP];  // kh_s . kh_t and kh_s . qh_t over s
        load_row<TP, true>(KKt + t * TP, kk);
        load_row<TP, true>(KQt + t * TP, kq);
        gamma *= g[t];
        float u = gamma * (pr[t] + pr[T + t]);            // gamma_t S_0 kh_t
        float o = gamma * (pr[2 * T + t] + pr[3 * T + t]);  // gamma_t S_0 qh_t
        float G = 1.f;
#pragma unroll
        for (int s = t - 1; s >= 0; --s) {  // G(s, t) = g_{s+1} ... g_t
            G *= g[s + 1];
            u = fmaf(G * kk[s], delta[s], u);
            o = fmaf(G * kq[s], delta[s], o);
        }
        delta[t] = be[t] * (v[t] - u);
        o = fmaf(kq[t], delta[t], o);
        const float ov = p.scale * o;
        if (p.out_bf16) {
            const __nv_bfloat16 ob = __float2bfloat16_rn(ov);
            ost[t] = __bfloat162float(ob);
            if (live) static_cast<__nv_bfloat16*>(p.o)[o0 + t * tok_out] = ob;
        } else {
            ost[t] = ov;
            if (live) static_cast<float*>(p.o)[o0 + t * tok_out] = ov;
        }
    }
}

// Replay commit: one row's coefficients c_s = G(s, L-1) delta_s (s < L, 0 beyond) from its P row, as its row of
// A2 = [c hi | c hi | c lo | 0] in bf16 pairs (hi = c rounded, lo = c - hi rounded; element 2j in the low half),
// to be multiplied by the B rows [kh hi; kh lo; kh hi].
template <int T, int NP, int K2>
__device__ __forceinline__ void row_coefficients(const float (&pr)[NP], const float* v, const float* gs,
                                                 const float* bs, const float* KKt, int L, uint32_t (&a2)[K2 / 2]) {
    constexpr int TP = (T + 3) & ~3;
    float delta[T];
    float gamma = 1.f;
#pragma unroll
    for (int t = 0; t < T; ++t) {
        delta[t] = 0.f;
        if (t < L) {
            gamma *= gs[t];
            float u = gamma * (pr[t] + pr[T + t]);  // gamma_t S_0 kh_t
            float G = 1.f;
#pragma unroll
            for (int s = t - 1; s >= 0; --s) {
                G *= gs[s + 1];
                u = fmaf(G * KKt[t * TP + s], delta[s], u);
            }
            delta[t] = bs[t] * (v[t] - u);
        }
    }
    float c[T];
    float G = 1.f;  // G(s, L-1), s = L-1, L-2, ...
#pragma unroll
    for (int s = T - 1; s >= 0; --s) {
        c[s] = 0.f;
        if (s < L) {
            c[s] = G * delta[s];
            G *= gs[s];
        }
    }
    float hi[T], lo[T];
#pragma unroll
    for (int s = 0; s < T; ++s) {
        hi[s] = __bfloat162float(__float2bfloat16_rn(c[s]));
        lo[s] = c[s] - hi[s];
    }
    auto col = [&](int i) -> float { return i < T ? hi[i] : (i < 2 * T ? hi[i - T] : (i < 3 * T ? lo[i - 2 * T] : 0.f)); };
#pragma unroll
    for (int i = 0; i < K2; i += 2) a2[i / 2] = bf16x2_bits(col(i), col(i + 1));
}

// Per-item inputs in registers, kept in their storage type until used (a conversion right after the load would
// wait for it): the q / k pieces of this lane (16 bytes of one vector per pass), v of row tid for the replay set
// and the verify set, and, on the last warp, a and b of one token (lanes 0..15: replay set, 16..31: verify set)
// with the head's A_log and dt_bias.  Each field is loaded for the next item right after its last use in the
// current one, so every load has about one item of lead time and none is waited for by a register copy.
template <int DK, typename InT, int kMode>
struct ItemRegs {
    static constexpr int MAXT = kMode == kModeReplayVerify ? kFusedMaxT : kChunkMaxT;
    static constexpr int VPASS = 4 * (32 / (DK / 8));  // vectors per pass of the group
    static constexpr int NVEC = (kMode != kModeVerify ? MAXT : 0) + (kMode != kModeReplay ? 2 * MAXT : 0);
    static constexpr int NPASS = (NVEC + VPASS - 1) / VPASS;
    uint4 raw[NPASS][Slice8<InT>::NC];
    InT vr[kMode != kModeVerify ? MAXT : 1];
    InT vv[kMode != kModeReplay ? MAXT : 1];
    uint32_t vz[kMode != kModeReplay ? MAXT : 1];  // z of the gated norm, raw (fp32 bits, or bf16 bits)
    InT a, b;
    float A_log, dt_bias;
};

// Gram matrix X[t][s] = x_s . y_t (x_s: rows s and T + s of the region, hi and lo; y_t: rows (yb) T + t and
// (yb + 1) T + t, hi and lo) on mma.sync, one warp: A rows 0..7 address x hi 0..7 and rows 8..15 x lo 0..7, B
// columns 8 nb .. 8 nb + 7 address block yb + nb; rows past T point at row 0 and their products are dropped.  The
// four products of a pair (hi.hi, hi.lo, lo.hi, lo.lo) then sit in one lane; two accumulation chains (even and
// odd k steps) halve the latency.  Stored transposed in rows of TP floats.
template <int DK>
__device__ __forceinline__ void gram_warp(uint32_t bbase, int BR, int T, int yb, float* out, int TP, int lane) {
    constexpr int KSTEPS = DK / 16;
    const int m = lane & 15;
    const int arow = m < 8 ? (m < T ? m : 0) : (m - 8 < T ? T + m - 8 : 0);
    const int jr = lane & 7;
    const int brow0 = jr < T ? yb * T + jr : 0, brow1 = jr < T ? (yb + 1) * T + jr : 0;
    float g[2][4], g2[2][4];
#pragma unroll
    for (int c = 0; c < 4; ++c) g[0][c] = g[1][c] = g2[0][c] = g2[1][c] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, c0, c1;
        ldsm_x4(bbase + sw128(BR, arow, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
        ldsm_x2(bbase + sw128(BR, brow0, 2 * ks + ((lane >> 3) & 1)), b0, b1);
        ldsm_x2(bbase + sw128(BR, brow1, 2 * ks + ((lane >> 3) & 1)), c0, c1);
        mma_bf16_16816((ks & 1) ? g2[0] : g[0], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816((ks & 1) ? g2[1] : g[1], a0, a1, a2, a3, c0, c1);
    }
    const int s_ = lane >> 2;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int t_ = 2 * (lane & 3) + e;
        if (s_ < T && t_ < T)
            out[t_ * TP + s_] = ((g[0][e] + g2[0][e]) + (g[1][e] + g2[1][e])) +
                                ((g[0][2 + e] + g2[0][2 + e]) + (g[1][2 + e] + g2[1][2 + e]));
    }
}

// Replay set, after its P MMA: every thread reads the P row of its state row from tensor memory and forms the
// row's coefficients; the group multiplies them into the tile on the tensor cores, each thread adds gamma_L S_0
// to its row and writes it over the stage, and PT stores the tile into the slot.  False: a wait ran out (the
// stage and the slot are left as they are).
template <int T, int DK, typename InT, int kMode, int NS>
__device__ __forceinline__ bool replay_rows(const CUtensorMap* tmap, uint32_t tmem, unsigned char* sm, uint32_t base,
                                            uint32_t stage, const float* v, const float* gs,
                                            const float* bs, const float* KK, int h, int HV, int row0, int slot, int L,
                                            int bar_id, uint32_t mma_bar, uint32_t& mphase) {
    using CS = ChunkPlan<DK, kMode, NS>;
    constexpr int PT = 64;
    constexpr int NP = CS::nr(T);
    constexpr int K2 = CS::rrows(T);
    const int tid = threadIdx.x & (kChunkGroupThreads - 1), warp = tid >> 5;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    float pr[NP];
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < NP; c += 16) tmem_ld16(lane_base + c, pr + c);
    tmem_wait_ld();
    uint32_t a2[K2 / 2];
    row_coefficients<T, NP, K2>(pr, v, gs, bs, KK, L, a2);
#pragma unroll
    for (int c = 0; c < K2 / 2; c += 8) tmem_st8(lane_base + CS::a2_col() + c, a2 + c);
    tmem_wait_st();
    float gamma = 1.f;
    for (int t = 0; t < L; ++t) gamma *= gs[t];
    tc_fence_before();
    group_sync(bar_id);  // every row's coefficients are in tensor memory, every P row has been read
    // D = A2 [kh hi; kh lo; kh hi] on the tensor cores: A2 from tensor memory, B = the replay rows read MN-major
    if (tid == PT) {
        tc_fence_after();
        const uint32_t idesc = umma_idesc_bf16(kChunkRows, DK) | (1u << 16);  // B MN-major
        const uint32_t brb = base + CS::br_off();
#pragma unroll
        for (int ks = 0; ks < K2 / 16; ++ks)
            umma_bf16_ta(tmem, tmem + CS::a2_col() + 8 * ks, umma_desc_sw128_mn(brb + 2048u * ks, K2 * 128u), idesc,
                         ks > 0 ? 1u : 0u);
        umma_commit(mma_bar);
    }
    const bool mok = mbar_wait_bounded(mma_bar, mphase, kChunkWaitPolls);
    mphase ^= 1u;
    if (group_sync_or(bar_id, !mok)) {  // the product never completed: leave the slot as it is
        if (tid == PT) mbar_wait_bounded(mma_bar, mphase ^ 1u, kChunkWaitPolls);
        return false;
    }
    tc_fence_after();
    // S_L = gamma S_0 + D, this thread's row, 32 columns at a time, rounded to bf16 over the stage
    unsigned char* srow = sm + (stage - base);
#pragma unroll 1
    for (int c32 = 0; c32 < DK / 32; ++c32) {
        float d[32];
        tmem_ld16(lane_base + 32 * c32, d);
        tmem_ld16(lane_base + 32 * c32 + 16, d + 16);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4* cp = reinterpret_cast<uint4*>(srow + sw128(kChunkRows, tid, 4 * c32 + q));
            const uint4 s0 = *cp;
            const uint32_t w[4] = {s0.x, s0.y, s0.z, s0.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = bf16x2_to_float2(w[e]);
                o[e] = bf16x2_bits(fmaf(gamma, f.x, d[8 * q + 2 * e]), fmaf(gamma, f.y, d[8 * q + 2 * e + 1]));
            }
            *cp = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    fence_proxy_async_smem();  // the rows written above, then the TMA store (and a verify MMA) read them
    tc_fence_before();
    group_sync(bar_id);
    if (tid == PT) {
#pragma unroll
        for (int j = 0; j < CS::NBOX; ++j) tma_store_3d(tmap, j * 64, row0, slot * HV + h, stage + j * CS::BOX_BYTES);
        bulk_commit_group();
    }
    return true;
}

// Verify set, after its P MMA: every thread reads the P row of its state row from tensor memory and runs the
// row's T x T recurrence, writing o.
template <int T, int DK, typename InT, int kMode, int NS>
__device__ __forceinline__ void verify_rows(const RecurrentParams& p, uint32_t tmem, const float* v,
                                            const uint32_t* z, float wrow, float* red, int bar_id,
                                            const float* gs, const float* bs, const float* KK, const float* KQ, int b,
                                            int h, int row0, int nrows) {
    using CS = ChunkPlan<DK, kMode, NS>;
    constexpr int NP = CS::vrows(T);
    const int tid = threadIdx.x & (kChunkGroupThreads - 1), warp = tid >> 5, lane = tid & 31;
    float pr[NP];
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < NP; c += 16) tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + c, pr + c);
    tmem_wait_ld();
    const bool live = tid < nrows;
    const int64_t o0 = ((int64_t)b * T * p.HV + h) * p.DV + row0 + tid;
    const int64_t tok_out = (int64_t)p.HV * p.DV;
    float ost[T];
    row_recurrence<T, NP>(p, pr, v, gs, bs, KK, KQ, live, o0, tok_out, ost);
    if (p.nz != nullptr) {
        // gated RMSNorm of the stored o over the DV rows of the head (this item holds all of them): sums of
        // squares per token over the warp (shuffles), then over the 4 warps (shared memory), in one order for
        // every thread
        float ss[T];
#pragma unroll
        for (int t = 0; t < T; ++t) ss[t] = live ? ost[t] * ost[t] : 0.f;
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
            for (int t = 0; t < T; ++t) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], m);
        if (lane == 0)
#pragma unroll
            for (int t = 0; t < T; ++t) red[warp * kChunkMaxT + t] = ss[t];
        group_sync(bar_id);
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float tot = (red[t] + red[kChunkMaxT + t]) + (red[2 * kChunkMaxT + t] + red[3 * kChunkMaxT + t]);
            const float inv_rms = 1.f / sqrtf(tot / (float)p.DV + p.neps);
            const float zt = p.nz_bf16 ? __uint_as_float(z[t] << 16) : __uint_as_float(z[t]);
            const float y = ost[t] * inv_rms * wrow * (zt / (1.f + expf(-zt)));
            if (live) {
                if (p.out_bf16)
                    static_cast<__nv_bfloat16*>(p.ny)[o0 + t * tok_out] = __float2bfloat16_rn(y);
                else
                    static_cast<float*>(p.ny)[o0 + t * tok_out] = y;
            }
        }
    }
}

// A kernel that allocates tensor memory runs one CTA per SM, so the CTA holds G groups of 4 warps, each an
// independent item pipeline (its own stages, B rows, Gram matrices, mbarriers, named barrier 1 + g and share of
// the tensor memory); group g of CTA c walks the items of virtual CTA g gridDim + c.
//   kModeVerify          p.q, p.k, p.v, p.a, p.b: T verify tokens; outputs o.
//   kModeReplay          p.k, p.v, p.a, p.b: the first steps[b] of T tokens, committed into the slot.
//   kModeReplayVerify    p.rk, p.rv, p.ra, p.rb: the first steps[b] of rT tokens committed into the slot, then
//                        p.q .. p.b: T verify tokens from the committed state (as stored, rounded to bf16).
template <int DK, typename InT, int kMode, int NS, int G>
__global__ void __launch_bounds__(kChunkGroupThreads * G, 1)
    gdn_verify_chunked_kernel(const RecurrentParams p, const __grid_constant__ CUtensorMap tmap, int n_items,
                              int per_cta) {
    using CS = ChunkPlan<DK, kMode, NS>;
    using QK = Slice8<InT>;
    using IR = ItemRegs<DK, InT, kMode>;
    constexpr bool kReplay = CS::kReplay, kVerify = CS::kVerify;
    constexpr int ROWS = kChunkRows;
    constexpr int KSTEPS = DK / 16;
    constexpr int LPV = DK / 8;        // lanes per q or k vector (8 columns each)
    constexpr int VPW = 32 / LPV;      // vectors per warp per pass
    constexpr int VPASS = 4 * VPW;     // vectors per group pass
    constexpr bool kEarly = !kReplay;  // verify only: a stage is refilled as soon as its MMA has completed
    static_assert(LPV <= 32, "DK");
    const int grp = threadIdx.x / kChunkGroupThreads;
    const int tid = threadIdx.x & (kChunkGroupThreads - 1), warp = tid >> 5, lane = tid & 31;
    const int bar_id = 1 + grp;  // named barrier 0 is the whole CTA's
    const int Tv = kVerify ? p.T : 0;                                       // verify tokens
    const int Tr = kMode == kModeReplay ? p.T : (kReplay ? p.rT : 0);       // replay tokens
    const int NRB = (p.DV + ROWS - 1) / ROWS;
    const int R = p.HV / p.HK;  // value heads per key head
    // virtual CTA grp * gridDim.x + blockIdx.x: with few items, group 0 of every CTA gets them first
    const int beg = (int)min((int64_t)n_items, ((int64_t)grp * gridDim.x + blockIdx.x) * per_cta);
    const int end = min(n_items, beg + per_cta);
    // roles in a group besides the shared work: warp 1 (and 0, and 3 in the combined mode) form the Gram
    // matrices, thread PT of warp 2 issues the TMA loads and stores and the MMAs (and alone waits on the tiles and
    // its bulk groups), warp 3 computes the gates; warp 0 of the CTA allocates the tensor memory for every group
    constexpr int PT = 64;
    constexpr int GATE_T0 = ROWS - 32;

    extern __shared__ unsigned char ch_smem[];
    const uint32_t raw_base = smem_u32(ch_smem);
    const uint32_t pad = ((raw_base + 1023u) & ~1023u) - raw_base;
    const uint32_t gbytes = CS::group_bytes(Tr, Tv);
    unsigned char* sm = ch_smem + pad + grp * gbytes;  // this group's part
    const uint32_t base = raw_base + pad + grp * gbytes;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ch_smem + pad + G * gbytes);
    const uint32_t ctl = base + CS::ctl_off(Tr, Tv);  // mbarrier of stage s at ctl + 8 s; the MMA's at ctl + 8 NS
    const uint32_t mma_bar = ctl + 8 * NS;
    volatile int* fail_flag = reinterpret_cast<volatile int*>(sm + CS::ctl_off(Tr, Tv) + 8 * (NS + 1));
    int* st_slot = reinterpret_cast<int*>(sm + CS::ctl_off(Tr, Tv) + 8 * (NS + 1) + 8);
    int* st_len = st_slot + NS;
    // B rows, swizzled: replay kh hi | kh lo | kh hi, then verify kh hi | kh lo | qh hi | qh lo; zero padding
    unsigned char* Br = sm + CS::br_off();
    unsigned char* Bv = sm + CS::bv_off(Tr);
    const uint32_t brb = base + CS::br_off(), bvb = base + CS::bv_off(Tr);
    const int RR = CS::rrows(Tr), VR = CS::vrows(Tv);
    float* gr = reinterpret_cast<float*>(sm + CS::s_off(Tr, Tv));  // replay g, beta
    float* br_ = gr + Tr;
    float* gv = br_ + Tr;  // verify g, beta
    float* bv_ = gv + Tv;
    float* KKr = reinterpret_cast<float*>(sm + CS::gram_off(Tr, Tv));
    float* KKv = KKr + Tr * CS::tp(Tr);
    float* KQv = KKv + Tv * CS::tp(Tv);
    float* red = reinterpret_cast<float*>(sm + CS::red_off(Tr, Tv));  // the gated norm's partial sums
    // the gated norm's weight of this thread's row (the norm is fused only when one item holds a whole head)
    const float wrow = (kVerify && p.nz != nullptr && tid < p.DV) ? p.nw[tid] : 0.f;

    // thread PT: start the tile of the item at `ip` (pool slot and token count loaded one issue earlier) into
    // stage s
    auto issue = [&](const ItemPos& ip, int slot, int L, int s) {
        const int h = ip.h, rb = ip.rb;
        const bool slot_ok = slot >= 0 && slot < p.num_slots;
        const bool len_ok = L >= 0 && L <= Tr;
        if (p.err != nullptr && h == 0 && rb == 0) {  // once per lane
            if (slot != -1 && !slot_ok)
                atomicOr(p.err, GDN_ERRBIT_INDEX);
            else if (kReplay && slot_ok && !len_ok)
                atomicOr(p.err, GDN_ERRBIT_ACCEPT_LEN);
        }
        // replay only: nothing to do for a lane without tokens to commit; combined: a bad length commits nothing
        const bool active = kMode == kModeReplay ? slot_ok && len_ok && L > 0 : slot_ok;
        st_slot[s] = active ? slot : -1;
        st_len[s] = kReplay && len_ok ? L : 0;
        bool issue_copy = active;
#ifdef GDN_TEST_MISSING_COPY
        // test build: the first item (lane 0, head 0, rows 0..) is never copied nor arrived on: its wait runs out
        if (ip.b == 0 && ip.h == 0 && ip.rb == 0) issue_copy = false;
#endif
        if (issue_copy) {
            const uint32_t bar = ctl + 8 * s;
            mbar_arrive_expect_tx(bar, CS::STAGE_BYTES);
#pragma unroll
            for (int j = 0; j < CS::NBOX; ++j)
                tma_load_3d(base + s * CS::STAGE_BYTES + j * CS::BOX_BYTES, &tmap, j * 64, rb * ROWS, slot * p.HV + h,
                            bar);
        }
    };
    // vectors of one item, numbered: replay k_0 .. k_{Tr-1}, then verify q_0 .. q_{Tv-1}, k_0 .. k_{Tv-1}
    const int NV = Tr + 2 * Tv;
    const int vj0 = warp * VPW + lane / LPV;  // this lane's vector in the first pass
    const int vc = lane % LPV;                // its columns [8 vc, 8 vc + 8): chunk vc of the row
    const InT* rk = static_cast<const InT*>(kMode == kModeReplay ? p.k : p.rk);
    const InT* rv = static_cast<const InT*>(kMode == kModeReplay ? p.v : p.rv);
    const InT* ra = static_cast<const InT*>(kMode == kModeReplay ? p.a : p.ra);
    const InT* rbp = static_cast<const InT*>(kMode == kModeReplay ? p.b : p.rb);
    auto vec_ptr = [&](int b, int hk, int j) -> const InT* {
        if (j < Tr) return rk + (((int64_t)b * Tr + j) * p.HK + hk) * DK + 8 * vc;
        j -= Tr;
        const int t = j < Tv ? j : j - Tv;
        return static_cast<const InT*>(j < Tv ? p.q : p.k) + (((int64_t)b * Tv + t) * p.HK + hk) * DK + 8 * vc;
    };
    auto load_qk = [&](const ItemPos& ip, bool need_qk, IR& r) {
#pragma unroll
        for (int ps = 0; ps < IR::NPASS; ++ps) {
            const int j = vj0 + ps * VPASS;
#pragma unroll
            for (int c = 0; c < QK::NC; ++c) r.raw[ps][c] = make_uint4(0, 0, 0, 0);
            if (need_qk && j < NV) QK::load_global(vec_ptr(ip.b, ip.hk, j), r.raw[ps]);
        }
    };
    auto load_v = [&](const ItemPos& ip, IR& r) {
        const int row = ip.rb * ROWS + tid;
        if constexpr (kReplay) {
            const InT* src = rv + ((int64_t)ip.b * Tr * p.HV + ip.h) * p.DV + row;
#pragma unroll
            for (int t = 0; t < IR::MAXT; ++t) {
                r.vr[t] = InT(0.f);
                if (t < Tr && row < p.DV) r.vr[t] = src[(int64_t)t * p.HV * p.DV];
            }
        }
        if constexpr (kVerify) {
            const int64_t off = ((int64_t)ip.b * Tv * p.HV + ip.h) * p.DV + row;
            const InT* src = static_cast<const InT*>(p.v) + off;
#pragma unroll
            for (int t = 0; t < IR::MAXT; ++t) {
                r.vv[t] = InT(0.f);
                r.vz[t] = 0u;
                if (t < Tv && row < p.DV) {
                    r.vv[t] = src[(int64_t)t * p.HV * p.DV];
                    if (p.nz != nullptr)
                        r.vz[t] = p.nz_bf16 ? (uint32_t)static_cast<const uint16_t*>(p.nz)[off + (int64_t)t * p.HV * p.DV]
                                            : static_cast<const uint32_t*>(p.nz)[off + (int64_t)t * p.HV * p.DV];
                }
            }
        }
    };
    // gate lanes of warp 3: 0..15 the replay set, 16..31 the verify set
    const int gt = tid - GATE_T0;
    const bool gate_r = kReplay && gt >= 0 && gt < Tr;
    const bool gate_v = kVerify && gt >= 16 && gt - 16 < Tv;
    auto load_ab = [&](const ItemPos& ip, IR& r) {
        r.a = r.b = InT(0.f);
        r.A_log = r.dt_bias = 0.f;
        if (gate_r || gate_v) {
            const int t = gate_r ? gt : gt - 16;
            const int64_t ab = ((int64_t)ip.b * (gate_r ? Tr : Tv) + t) * p.HV + ip.h;
            r.a = (gate_r ? ra : static_cast<const InT*>(p.a))[ab];
            r.b = (gate_r ? rbp : static_cast<const InT*>(p.b))[ab];
            r.A_log = p.A_log[ip.h];
            r.dt_bias = p.dt_bias[ip.h];
        }
    };

    ItemPos pos = ItemPos::of(beg, NRB, p.HV, R);  // the current item
    ItemPos ipos = pos;  // thread PT: the next item to issue (number nis), with its slot and token count
    int nis = beg;
    int islot = 0, ilen = 0;
    auto issue_next = [&](int s) {  // thread PT: issue item nis into stage s, then look up the one after it
        issue(ipos, islot, ilen, s);
        ipos.next(NRB, p.HV, R);
        if (++nis < end) {
            islot = p.indices[ipos.b];
            ilen = kReplay ? p.steps[ipos.b] : 0;
        }
    };
    // tensor-memory columns of the CTA: a power of 2 covering every group's share
    constexpr uint32_t kCols = G * CS::tmem_cols() <= 32    ? 32u
                               : G * CS::tmem_cols() <= 64  ? 64u
                               : G * CS::tmem_cols() <= 128 ? 128u
                               : G * CS::tmem_cols() <= 256 ? 256u
                                                            : 512u;
    static_assert(G * CS::tmem_cols() <= 512, "tensor memory of the groups");
    if (threadIdx.x < 32) tmem_alloc(smem_u32(tmem_slot), kCols);
    if (tid == PT && beg < end) {
        for (int s = 0; s <= NS; ++s) mbar_init(ctl + 8 * s, 1);
        fence_mbar_init();
        *fail_flag = 0;
        islot = p.indices[ipos.b];
        ilen = kReplay ? p.steps[ipos.b] : 0;
        for (int j = 0; j < (kEarly ? NS : NS - 1) && nis < end; ++j) issue_next(j);
    }
    // the padding rows of B stay zero (the products with them are never used, and must be finite)
    for (int i2 = 3 * Tr * (DK / 8) + tid; i2 < RR * (DK / 8); i2 += ROWS)
        *reinterpret_cast<uint4*>(Br + sw128(RR, i2 / (DK / 8), i2 % (DK / 8))) = make_uint4(0, 0, 0, 0);
    for (int i2 = 4 * Tv * (DK / 8) + tid; i2 < VR * (DK / 8); i2 += ROWS)
        *reinterpret_cast<uint4*>(Bv + sw128(VR, i2 / (DK / 8), i2 % (DK / 8))) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();  // the padding rows are read by the tensor cores too
    IR in;  // the current item's inputs (each field refilled for the next item after its last use)
    if (beg < end) {
        load_qk(pos, true, in);
        load_v(pos, in);
        load_ab(pos, in);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tmem = tmem_base + CS::tmem_cols() * grp;  // this group's columns

    uint32_t phase = 0;   // bit s: parity of the next completion of stage s
    uint32_t mphase = 0;  // parity of the next completion of the MMA barrier
    int prev_b = -1, prev_hk = -1;
    bool failed = false;
    for (int i = 0, it = beg; it < end; ++i, ++it) {
        const int st = i % NS;
        const int b = pos.b, h = pos.h, rb = pos.rb;
        const int hk = pos.hk;
        const int row0 = rb * ROWS;
        const int nrows = min(ROWS, p.DV - row0);
        const int slot = st_slot[st];
        const int L = st_len[st];
        const bool active = slot >= 0;
        const bool replay_now = kReplay && active && L > 0;
        const bool reuse = b == prev_b && hk == prev_hk;  // same lane and key head: q, k, Gram still in place
        prev_b = b;
        prev_hk = hk;
        ItemPos npos = pos;
        npos.next(NRB, p.HV, R);

        if (active && !reuse) {
            // token prologue: normalise q and k into bf16 hi + lo rows of B
#pragma unroll
            for (int pass = 0; pass < IR::NPASS; ++pass) {
                if (pass * VPASS >= NV) break;
                const int j = vj0 + pass * VPASS;
                float2 x[4];
                QK::unpack(in.raw[pass], x);
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) ss = fmaf(x[e].x, x[e].x, fmaf(x[e].y, x[e].y, ss));
#pragma unroll
                for (int m = 1; m < LPV; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
                if (j < NV) {
                    const float rn = rsqrtf(ss + p.l2_eps);
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float f0 = x[e].x * rn, f1 = x[e].y * rn;
                        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(f0, f1);
                        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(f0 - __low2float(hi2), f1 - __high2float(hi2));
                        hw[e] = *reinterpret_cast<const uint32_t*>(&hi2);
                        lw[e] = *reinterpret_cast<const uint32_t*>(&lo2);
                    }
                    const uint4 hv = make_uint4(hw[0], hw[1], hw[2], hw[3]), lv = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    if (j < Tr) {  // replay k_j: rows j (hi), Tr + j (lo), 2 Tr + j (hi again)
                        *reinterpret_cast<uint4*>(Br + sw128(RR, j, vc)) = hv;
                        *reinterpret_cast<uint4*>(Br + sw128(RR, Tr + j, vc)) = lv;
                        *reinterpret_cast<uint4*>(Br + sw128(RR, 2 * Tr + j, vc)) = hv;
                    } else {  // verify q_t: rows 2 Tv + t, 3 Tv + t; k_t: rows t, Tv + t
                        const int jj = j - Tr;
                        const int t = jj < Tv ? jj : jj - Tv;
                        const int hi_row = jj < Tv ? 2 * Tv + t : t;
                        *reinterpret_cast<uint4*>(Bv + sw128(VR, hi_row, vc)) = hv;
                        *reinterpret_cast<uint4*>(Bv + sw128(VR, hi_row + Tv, vc)) = lv;
                    }
                }
            }
            fence_proxy_async_smem();  // B is written here and read by the tensor cores' MMA
        }
        if (it + 1 < end) load_qk(npos, !(npos.b == b && npos.hk == hk), in);
        tc_fence_before();
        group_sync(bar_id);
        // replay modes: the refill of the stage the last item used, once its store has read it
        if (!kEarly && tid == PT && nis < end && nis == it + NS - 1) {
            bulk_wait_read_all();
            issue_next((i + NS - 1) % NS);
        }
        if (active && (gate_r || gate_v)) {
            float* gd = gate_r ? gr + gt : gv + (gt - 16);
            gd[0] = gate(in.A_log, to_f32(in.a), in.dt_bias);
            gd[gate_r ? Tr : Tv] = sigmoid(to_f32(in.b));
        }
        if (it + 1 < end) load_ab(npos, in);
        if (active && !reuse) {
            if (kMode == kModeVerify) {
                if (warp == 1) gram_warp<DK>(bvb, VR, Tv, 0, KKv, CS::tp(Tv), lane);
                if (warp == 0) gram_warp<DK>(bvb, VR, Tv, 2, KQv, CS::tp(Tv), lane);
            } else if (kMode == kModeReplay) {
                if (warp == 1) gram_warp<DK>(brb, RR, Tr, 0, KKr, CS::tp(Tr), lane);
            } else {
                if (warp == 1) gram_warp<DK>(brb, RR, Tr, 0, KKr, CS::tp(Tr), lane);
                if (warp == 0) gram_warp<DK>(bvb, VR, Tv, 2, KQv, CS::tp(Tv), lane);
                if (warp == 3) gram_warp<DK>(bvb, VR, Tv, 0, KKv, CS::tp(Tv), lane);
            }
        }
        // the first MMA, issued by PT once the tile has landed: S_0 [kh hi | kh lo] of the replay set, or (nothing
        // to commit) S_0 [kh hi | kh lo | qh hi | qh lo] of the verify set
        if (active && tid == PT) {
            if (mbar_wait_bounded(ctl + 8 * st, (phase >> st) & 1u, kChunkWaitPolls)) {
                tc_fence_after();
                const uint32_t bb = replay_now ? brb : bvb;
                const uint32_t box = (uint32_t)(replay_now ? RR : VR) * 128u;
                const uint32_t idesc = umma_idesc_bf16(ROWS, replay_now ? CS::nr(Tr) : VR);
                const uint32_t stage = base + st * CS::STAGE_BYTES;
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    const uint32_t koff = (uint32_t)((ks & 3) * 32);  // 16 columns further inside the 128-byte span
                    umma_bf16(tmem, umma_desc_sw128(stage + (uint32_t)(ks >> 2) * CS::BOX_BYTES + koff),
                              umma_desc_sw128(bb + (uint32_t)(ks >> 2) * box + koff), idesc, ks > 0 ? 1u : 0u);
                }
                umma_commit(mma_bar);
            } else {
                *fail_flag = 1;
                mbar_arrive(mma_bar);  // releases the other threads' wait on the MMA; they see the flag
            }
        }
        if (active) phase ^= 1u << st;
        bool mok = true;
        if (active) {
            mok = mbar_wait_bounded(mma_bar, mphase, kChunkWaitPolls);
            mphase ^= 1u;
        }
        // every thread has seen the MMA complete (so the stage and B are read); the Gram matrices and the gates
        // are in place
        if (group_sync_or(bar_id, !mok || (active && *fail_flag != 0))) {
            failed = true;
            if (tid == PT) {
                if (p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_TIMEOUT);
                // drain what is in flight before leaving: this item's tile and MMA, and the tiles issued ahead
                if (active) {
                    mbar_wait_bounded(ctl + 8 * st, ((phase >> st) & 1u) ^ 1u, kChunkWaitPolls);
                    mbar_wait_bounded(mma_bar, mphase ^ 1u, kChunkWaitPolls);
                }
                for (int j = 1; j < NS && it + j < nis; ++j) {
                    const int s2 = (i + j) % NS;
                    if (st_slot[s2] >= 0) mbar_wait_bounded(ctl + 8 * s2, (phase >> s2) & 1u, kChunkWaitPolls);
                }
                if (kReplay) bulk_wait_all();
            }
            break;
        }
        // verify only: the stage is free as soon as its MMA has completed
        if (kEarly && tid == PT && nis < end) issue_next(st);

        float vrr[IR::MAXT], vrv[IR::MAXT];
        uint32_t zr[IR::MAXT];  // this item's z before the next item's loads replace it
#pragma unroll
        for (int t = 0; t < IR::MAXT; ++t) {
            vrr[t] = kReplay ? to_f32(in.vr[kReplay ? t : 0]) : 0.f;
            vrv[t] = kVerify ? to_f32(in.vv[kVerify ? t : 0]) : 0.f;
            zr[t] = kVerify ? in.vz[kVerify ? t : 0] : 0u;
        }
        if (it + 1 < end) load_v(npos, in);
        if (active) {
            const uint32_t stage = base + st * CS::STAGE_BYTES;
            bool ok = true;
            if constexpr (kReplay) if (replay_now) {
                // the write-back reads the tile itself: each thread acquires the landed copy (its wait ends at
                // once: PT saw the phase complete)
                mbar_wait_bounded(ctl + 8 * st, ((phase >> st) & 1u) ^ 1u, kChunkWaitPolls);
#define GDN_REPLAY_ROWS(TT)                                                                                      \
    ok = replay_rows<TT, DK, InT, kMode, NS>(&tmap, tmem, sm, base, stage, vrr, gr, br_, KKr, h, p.HV, row0, slot, L, \
                                             bar_id, mma_bar, mphase)
                // token counts above MAXT never reach this kernel (the launcher's range)
                switch (Tr) {
                case 1: GDN_REPLAY_ROWS(1); break;
                case 2: GDN_REPLAY_ROWS(2); break;
                case 3: GDN_REPLAY_ROWS(3); break;
                case 4: GDN_REPLAY_ROWS(4); break;
                case 5: GDN_REPLAY_ROWS(IR::MAXT < 5 ? IR::MAXT : 5); break;
                case 6: GDN_REPLAY_ROWS(IR::MAXT < 6 ? IR::MAXT : 6); break;
                case 7: GDN_REPLAY_ROWS(IR::MAXT < 7 ? IR::MAXT : 7); break;
                default: GDN_REPLAY_ROWS(IR::MAXT); break;
                }
#undef GDN_REPLAY_ROWS
                if (kVerify && ok) {
                    // the verify set's MMA on the committed state, from the rows just written over the stage
                    if (tid == PT) {
                        tc_fence_after();
                        const uint32_t idesc = umma_idesc_bf16(ROWS, VR);
#pragma unroll
                        for (int ks = 0; ks < KSTEPS; ++ks) {
                            const uint32_t koff = (uint32_t)((ks & 3) * 32);
                            umma_bf16(tmem, umma_desc_sw128(stage + (uint32_t)(ks >> 2) * CS::BOX_BYTES + koff),
                                      umma_desc_sw128(bvb + (uint32_t)(ks >> 2) * (uint32_t)VR * 128u + koff), idesc,
                                      ks > 0 ? 1u : 0u);
                        }
                        umma_commit(mma_bar);
                    }
                    const bool vok = mbar_wait_bounded(mma_bar, mphase, kChunkWaitPolls);
                    mphase ^= 1u;
                    if (group_sync_or(bar_id, !vok)) {
                        if (tid == PT) mbar_wait_bounded(mma_bar, mphase ^ 1u, kChunkWaitPolls);
                        ok = false;
                    }
                }
            }
            if constexpr (kVerify) if (ok) {
#define GDN_VERIFY_ROWS(TT) \
    verify_rows<TT, DK, InT, kMode, NS>(p, tmem, vrv, zr, wrow, red, bar_id, gv, bv_, KKv, KQv, b, h, row0, nrows)
                switch (Tv) {
                case 1: GDN_VERIFY_ROWS(1); break;
                case 2: GDN_VERIFY_ROWS(2); break;
                case 3: GDN_VERIFY_ROWS(3); break;
                case 4: GDN_VERIFY_ROWS(4); break;
                case 5: GDN_VERIFY_ROWS(IR::MAXT < 5 ? IR::MAXT : 5); break;
                case 6: GDN_VERIFY_ROWS(IR::MAXT < 6 ? IR::MAXT : 6); break;
                case 7: GDN_VERIFY_ROWS(IR::MAXT < 7 ? IR::MAXT : 7); break;
                default: GDN_VERIFY_ROWS(IR::MAXT); break;
                }
#undef GDN_VERIFY_ROWS
            }
            if (!ok) {  // a wait ran out inside: report it and drain the tiles issued ahead
                failed = true;
                if (tid == PT) {
                    if (p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_TIMEOUT);
                    for (int j = 1; j < NS && it + j < nis; ++j) {
                        const int s2 = (i + j) % NS;
                        if (st_slot[s2] >= 0) mbar_wait_bounded(ctl + 8 * s2, (phase >> s2) & 1u, kChunkWaitPolls);
                    }
                    bulk_wait_all();
                }
                break;
            }
        }
        pos = npos;
    }
    if (kReplay && !failed && tid == PT) bulk_wait_all();
    // every group's tensor-memory reads are complete before the allocation is released
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(tmem_base, kCols);
}

// ---- host side ------------------------------------------------------------------------------------------------
// The bf16 pool as a 3-D tensor [num_slots * HV][DV][DK]; box = (64 columns, 128 rows, 1), 128-byte swizzle.
template <int DK>
cudaError_t encode_pool_map(CUtensorMap* map, void* pool, const RecurrentParams& p) {
    const EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)p.DV, (cuuint64_t)p.num_slots * (cuuint64_t)p.HV};
    const cuuint64_t strides[2] = {(cuuint64_t)DK * 2, (cuuint64_t)p.DV * DK * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kChunkRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pool, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// TMA stages per CTA (state tiles in flight or being read by the MMA)
#ifndef GDN_CHUNK_STAGES
#define GDN_CHUNK_STAGES 2
#endif
constexpr int kChunkStages = GDN_CHUNK_STAGES;
// verify alone may run on other settings (its stage is free once its P product has completed): stages and the most
// groups per CTA
#ifndef GDN_VERIFY_STAGES
#define GDN_VERIFY_STAGES GDN_CHUNK_STAGES
#endif
#ifndef GDN_VERIFY_GROUPS
#define GDN_VERIFY_GROUPS 3
#endif
template <int kMode>
constexpr int chunk_stages() {
    return kMode == kModeVerify ? GDN_VERIFY_STAGES : kChunkStages;
}
constexpr int kChunkCachedDevices = 64;  // devices whose launch settings are cached
constexpr uint32_t kChunkMaxSmem = 227 * 1024;  // dynamic shared memory a CTA may open

// groups per CTA: as many as the shared memory of T = 8 (in every token set of the mode) and the tensor memory
// allow, up to kChunkMaxGroups (verify alone: GDN_VERIFY_GROUPS)
template <int DK, int kMode, int NS>
constexpr int chunk_groups() {
    using CS = ChunkPlan<DK, kMode, NS>;
    for (int g = kMode == kModeVerify ? GDN_VERIFY_GROUPS : kChunkMaxGroups; g > 1; --g)
        if (CS::max_bytes(g) <= kChunkMaxSmem && g * CS::tmem_cols() <= 512) return g;
    return 1;
}

// grid = min(items, SMs x resident CTAs) CTAs of G groups, each group a contiguous range of items
template <int DK, typename InT, int kMode, int G>
cudaError_t launch_chunked_groups(const RecurrentParams& p, int B, int Tr, int Tv, cudaStream_t s) {
    constexpr int NS = chunk_stages<kMode>();
    using CS = ChunkPlan<DK, kMode, NS>;
    auto kernel = gdn_verify_chunked_kernel<DK, InT, kMode, NS, G>;
    const uint32_t smem = CS::bytes(Tr, Tv, G);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // Launch caches shared by every calling thread, one entry per device: the shared-memory opening is a
    // per-device attribute of the function, and occupancy may differ between devices.  A repeated first call
    // only repeats the same queries; devices beyond the table are queried on every call.
    static std::atomic<int> attr_bytes[kChunkCachedDevices];                 // bytes opened on each device
    static std::atomic<int> occ_cache[kChunkCachedDevices][(kChunkMaxT + 1) * (kChunkMaxT + 1)];  // zero (static)
    const bool cached = dev >= 0 && dev < kChunkCachedDevices;
    if (!cached || (int)smem > attr_bytes[dev].load(std::memory_order_relaxed)) {
        const int most = (int)std::min<uint32_t>(CS::max_bytes(G), kChunkMaxSmem);
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
        if (e != cudaSuccess) return e;
        if (cached) attr_bytes[dev].store(most, std::memory_order_relaxed);
    }
    const int okey = Tr * (kChunkMaxT + 1) + Tv;
    int occ = cached ? occ_cache[dev][okey].load(std::memory_order_relaxed) : 0;
    if (occ == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kChunkGroupThreads * G, smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        if (cached) occ_cache[dev][okey].store(occ, std::memory_order_relaxed);
    }
    CUtensorMap map;
    e = encode_pool_map<DK>(&map, kMode == kModeVerify ? const_cast<void*>(p.pool_in) : p.pool_out, p);
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)B * p.HV * ((p.DV + kChunkRows - 1) / kChunkRows);
    if (items > INT32_MAX) return cudaErrorInvalidValue;
    const int64_t ctas = std::min<int64_t>(items, (int64_t)sms * occ);
    const int64_t vctas = std::min<int64_t>(items, ctas * G);
    const int per_cta = (int)((items + vctas - 1) / vctas);
    kernel<<<(int)ctas, kChunkGroupThreads * G, smem, s>>>(p, map, (int)items, per_cta);
    return cudaGetLastError();
}

// The group count: as many as the largest token counts of the mode allow.
template <int DK, typename InT, int kMode>
cudaError_t launch_chunked(const RecurrentParams& p, int B, cudaStream_t s) {
    constexpr int NS = chunk_stages<kMode>();
    constexpr int G = chunk_groups<DK, kMode, NS>();
    using CS = ChunkPlan<DK, kMode, NS>;
    static_assert(CS::max_bytes(G) <= kChunkMaxSmem, "shared memory of one group");
    const int Tv = kMode == kModeReplay ? 0 : p.T;
    const int Tr = kMode == kModeVerify ? 0 : (kMode == kModeReplay ? p.T : p.rT);
    return launch_chunked_groups<DK, InT, kMode, G>(p, B, Tr, Tv, s);
}

}  // namespace gdn
