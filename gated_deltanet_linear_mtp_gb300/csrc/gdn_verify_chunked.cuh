// gdn_verify_chunked.cuh -- MTP verify without intermediate states, and the replay commit, in chunked form on
// the tensor cores; persistent CTAs stream the state tiles through a ring of TMA stages.
//
// When nothing needs the states S_1..S_T themselves, the recurrence can be unrolled.  Writing
// gamma_t = g_1 ... g_t, G(s,t) = g_{s+1} ... g_t (G(t,t) = 1) and delta_t = beta_t (v_t - u_t),
// S_t = g_t S_{t-1} + delta_t kh_t^T unrolls to
//     S_t = gamma_t S_0 + sum_{s<=t} G(s,t) delta_s kh_s^T,
// so for every state row
//     u_t = g_t S_{t-1} kh_t = gamma_t (S_0 kh_t) + sum_{s<t}  G(s,t) (kh_s . kh_t) delta_s
//     o_t = S_t qh_t         = gamma_t (S_0 qh_t) + sum_{s<=t} G(s,t) (kh_s . qh_t) delta_s .
// The only per-element work is the contraction S_0 [kh_1..kh_T qh_1..qh_T], a (rows x DK) x (DK x 2T)
// product: it runs on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) with S_0 exact in
// bf16 and kh, qh split into bf16 hi + lo parts (4T columns), which keeps about 16 significant bits of
// kh and qh.  The T x T Gram matrices kh.kh and kh.qh are formed on the tensor cores from the same hi + lo
// rows, and each row's small triangular recurrence runs in fp32 registers, one thread per row.
//
// Two modes, for bf16 state pools and T <= 8 (the launcher's choice):
//   verify (kCommit = false)   outputs o only: no intermediate states, no write-back;
//   replay commit (kCommit)    the first L = steps[b] tokens, no outputs, and the state after them,
//                              S_L = gamma_L S_0 + sum_{s<L} G(s, L-1) delta_s kh_s^T, written back into the
//                              slot (kh only: 2T columns, one Gram matrix); the rank-L update runs on the
//                              tensor cores too.
//
// Work item = 128 state rows of one (lane, value head); items are numbered row block fastest, then value
// head, then lane, and each CTA (4 warps, warp w owning rows [32w, 32w + 32)) takes a contiguous range of
// them.  One thread (PT) keeps NS - 1 state tiles in flight ahead of the item being computed: one 3-D TMA
// tensor load per 64-column box into a 1024-byte aligned stage, rows past DV filled with zeros, 16-byte chunks
// swizzled within each 128-byte line so that the ldmatrix reads of the MMA are conflict-free.  q, k, v, a
// and b of the next item are loaded into registers while the current one is computed, and consecutive
// items of one key head reuse its normalised q, k and Gram matrices.  The replay commit rewrites the tile
// in place and stores it with a TMA tensor store (rows past DV are not written).
#pragma once

#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "gdn_common.cuh"

namespace gdn {

constexpr int kChunkRows = 128;  // state rows per item: 4 warps x 32
constexpr int kChunkThreads = 128;
constexpr int kChunkMaxT = 8;
constexpr uint32_t kChunkWaitPolls = GDN_WAIT_POLLS;

// Shared-memory plan of one CTA, as byte offsets from a 1024-byte aligned base.
template <int DK, bool kCommit, int NS>
struct ChunkPlan {
    static constexpr uint32_t SWZ = DK * 2 < 128 ? DK * 2 : 128;  // swizzle span = bytes of one box row
    static constexpr int BOX_COLS = SWZ / 2;
    static constexpr int NBOX = DK / BOX_COLS;
    static constexpr uint32_t BOX_BYTES = kChunkRows * SWZ;
    static constexpr uint32_t STAGE_BYTES = kChunkRows * DK * 2;
    static constexpr uint32_t ROW_BYTES = DK * 2 + 16;  // padded bf16 row of B
    // columns of P: kh hi, kh lo (and qh hi, qh lo in verify mode), T each
    __host__ __device__ static int ncols(int T) { return kCommit ? 2 * T : 4 * T; }
    __host__ __device__ static int b_rows(int T) { return ((ncols(T) + 7) / 8) * 8; }  // whole n8 tiles
    // fp32 row stride of P: verify with even T pads rows to 4T + 4 floats, so that a thread reads its row with
    // float4 loads (T + 1 odd keeps 8 consecutive rows on 8 distinct 16-byte bank groups); otherwise + 1
    __host__ __device__ static int p_stride(int T) { return (!kCommit && T % 2 == 0) ? 4 * T + 4 : ncols(T) + 1; }
    __host__ __device__ static int gram_stride(int T) { return (T + 3) & ~3; }  // padded row of the Gram matrices
    // Where a warp's 32 rows of P go (verify; the replay commit has a region of its own):
    //   0  over the warp's own 32 rows of the stage's first box, once its MMAs are done (no CTA barrier);
    //   1  likewise over its own rows of the first two boxes, 16 P rows in each (rows too long for one box);
    //   2  over the whole stage, after a CTA barrier (every warp's MMAs done);
    //   3  a region of its own.
    __host__ __device__ static int p_mode(int T) {
        if (kCommit) return 3;
        const uint32_t row = (uint32_t)p_stride(T) * 4;
        if (row <= SWZ) return 0;
        if (NBOX >= 2 && 16u * row <= 32u * SWZ) return 1;
        if ((uint32_t)kChunkRows * row <= STAGE_BYTES) return 2;
        return 3;
    }
    __host__ __device__ static uint32_t b_off() { return NS * STAGE_BYTES; }
    // replay commit: the coefficient tile A2 = [c hi | c lo | c hi | 0] (bf16, rows padded by 16 bytes)
    __host__ __device__ static int a2_cols(int T) { return 3 * T <= 16 ? 16 : 32; }
    __host__ __device__ static uint32_t a2_stride(int T) { return (uint32_t)a2_cols(T) * 2 + 16; }
    // replay commit: bytes of one warp's P rows, later covered by its A2 rows
    __host__ __device__ static uint32_t warp_region(int T) {
        const uint32_t pw = 32u * p_stride(T) * 4, aw = 32u * a2_stride(T);
        return pw > aw ? pw : aw;
    }
    __host__ __device__ static uint32_t p_off(int T) { return b_off() + (uint32_t)b_rows(T) * ROW_BYTES; }
    __host__ __device__ static uint32_t s_off(int T) {
        if (kCommit) return p_off(T) + 4u * warp_region(T);
        return p_off(T) + (p_mode(T) < 3 ? 0u : (uint32_t)kChunkRows * p_stride(T) * 4);
    }
    // g, beta (T each), then the Gram matrices, transposed (row t holds kh_s . kh_t, kh_s . qh_t over s)
    __host__ __device__ static uint32_t gram_off(int T) { return s_off(T) + ((8u * T + 15u) & ~15u); }
    // NS mbarriers, then per stage the pool slot (-1: nothing loaded) and the token count of its item
    __host__ __device__ static uint32_t ctl_off(int T) { return gram_off(T) + 2u * T * gram_stride(T) * 4; }
    __host__ __device__ static uint32_t bytes(int T) { return ctl_off(T) + NS * 16 + 1024; }  // + alignment slack
};

// Byte offset of the 16-byte chunk c of row r in a stage: box c / CPB, and inside the box the chunk index
// XORed with bits 7.. of its linear offset (the TMA 32 / 64 / 128-byte swizzle patterns).
template <int DK>
__device__ __forceinline__ uint32_t swz_off(int r, int c) {
    constexpr uint32_t SWZ = DK * 2 < 128 ? DK * 2 : 128;
    constexpr int CPB = SWZ / 16;
    const uint32_t lin = (uint32_t)r * SWZ + (uint32_t)(c % CPB) * 16;
    return (uint32_t)(c / CPB) * (kChunkRows * SWZ) + (lin ^ (((lin >> 7) & (CPB - 1)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void stsm_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h2);
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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

// One row's T x T recurrence (T fixed at compile time, so delta stays in registers).  Pr: the row of P,
// [S_0 kh hi | S_0 kh lo | S_0 qh hi | S_0 qh lo]; v: the row's v per token; KKt, KQt: the transposed Gram
// matrices, rows of TP = gram_stride(T) floats.
template <int T>
__device__ __forceinline__ void row_recurrence(const RecurrentParams& p, const float* Pr, const float (&v)[kChunkMaxT],
                                               const float* gs, const float* bs, const float* KKt, const float* KQt,
                                               bool live, int64_t o0, int64_t tok_out) {
    constexpr int TP = (T + 3) & ~3;
    float pr[4 * T];
    load_row<4 * T, T % 2 == 0>(Pr, pr);
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
        if (live) {
            const float ov = p.scale * o;
            if (p.out_bf16)
                static_cast<__nv_bfloat16*>(p.o)[o0 + t * tok_out] = __float2bfloat16_rn(ov);
            else
                static_cast<float*>(p.o)[o0 + t * tok_out] = ov;
        }
    }
}

// Replay commit: one row's coefficients c_s = G(s, L-1) delta_s (s < L, 0 beyond), read from its P row and,
// after the warp's __syncwarp, written as its row of A2 = [c hi | c lo | c hi | 0] in bf16 (hi = c rounded,
// lo = c - hi rounded), to be multiplied by [kh hi; kh hi; kh lo].
template <int T>
__device__ __forceinline__ void row_coefficients(const float* Pr, const float (&v)[kChunkMaxT], const float* gs,
                                                 const float* bs, const float* KKt, int L, unsigned char* a2row) {
    constexpr int TP = (T + 3) & ~3;
    float delta[T];
    float gamma = 1.f;
    float a[T];
#pragma unroll
    for (int t = 0; t < T; ++t) a[t] = Pr[t] + Pr[T + t];  // S_0 kh_t
#pragma unroll
    for (int t = 0; t < T; ++t) {
        delta[t] = 0.f;
        if (t < L) {
            gamma *= gs[t];
            float u = gamma * a[t];
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
    constexpr int W = 3 * T <= 16 ? 16 : 32;
    auto col = [&](int i) -> float { return i < T ? hi[i] : (i < 2 * T ? lo[i - T] : (i < 3 * T ? hi[i - 2 * T] : 0.f)); };
    __syncwarp();  // every lane of the warp has read its P row
    uint32_t w[W / 2];
#pragma unroll
    for (int i = 0; i < W; i += 2) w[i / 2] = bf16x2_bits(col(i), col(i + 1));
#pragma unroll
    for (int q = 0; q < W / 8; ++q)
        *reinterpret_cast<uint4*>(a2row + 16 * q) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// Per-item registers loaded one item ahead, kept in their storage type until used (a conversion right after
// the load would wait for it): q / k (this lane's 16-byte pieces of every vector pass), v of row tid, and, on
// the last warp, a and b of token tid - (128 - 32) with the head's A_log and dt_bias.
template <int DK, typename InT, bool kCommit>
struct ItemRegs {
    static constexpr int VPASS = 4 * (32 / (DK / 8));
    static constexpr int NPASS = ((kCommit ? 1 : 2) * kChunkMaxT + VPASS - 1) / VPASS;
    uint4 raw[NPASS][Slice8<InT>::NC];
    InT v[kChunkMaxT];
    InT a, b;
    float A_log, dt_bias;
};


template <int DK, typename InT, bool kCommit, int NS>
__global__ void __launch_bounds__(kChunkThreads, 3) gdn_verify_chunked_kernel(const RecurrentParams p,
                                                                          const __grid_constant__ CUtensorMap tmap,
                                                                          int n_items, int per_cta) {
    using CS = ChunkPlan<DK, kCommit, NS>;
    using QK = Slice8<InT>;
    constexpr int ROWS = kChunkRows;
    constexpr int KSTEPS = DK / 16;
    constexpr int LPV = DK / 8;       // lanes per q or k vector (8 columns each)
    constexpr int VPW = 32 / LPV;     // vectors per warp per pass
    constexpr int VPASS = 4 * VPW;    // vectors per CTA pass
    constexpr int CPR = DK / 8;       // 16-byte chunks per state row
    static_assert(DK % 16 == 0 && LPV <= 32 && ROWS % CPR == 0, "DK");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T;
    const int NRB = (p.DV + ROWS - 1) / ROWS;
    const int R = p.HV / p.HK;  // value heads per key head
    const int beg = blockIdx.x * per_cta;
    const int end = min(n_items, beg + per_cta);
    if (beg >= end) return;
    // roles besides the shared work: warp 1 forms the Gram matrices, thread PT of warp 2 issues the TMA
    // loads and stores (and alone waits on its bulk groups), warp 3 computes the gates
    constexpr int PT = 64;
    constexpr int GATE_T0 = ROWS - 32;

    extern __shared__ unsigned char ch_smem[];
    const uint32_t raw_base = smem_u32(ch_smem);
    const uint32_t pad = ((raw_base + 1023u) & ~1023u) - raw_base;
    unsigned char* sm = ch_smem + pad;
    const uint32_t base = raw_base + pad;
    const uint32_t ctl = base + CS::ctl_off(T);  // mbarrier of stage s at ctl + 8 s
    int* st_slot = reinterpret_cast<int*>(sm + CS::ctl_off(T) + NS * 8);
    int* st_len = st_slot + NS;
    unsigned char* Bs = sm + CS::b_off();  // rows: k hi (T) | k lo (T) | q hi (T) | q lo (T) | zeros
    float* gs = reinterpret_cast<float*>(sm + CS::s_off(T));
    float* bs = gs + T;
    const int TP = CS::gram_stride(T);
    float* KK = reinterpret_cast<float*>(sm + CS::gram_off(T));  // transposed: KK[t * TP + s] = kh_s . kh_t
    float* KQ = KK + T * TP;                                     // transposed: KQ[t * TP + s] = kh_s . qh_t

    // thread PT: start the tile of the item at `ip` (pool slot and token count loaded one issue earlier) into
    // stage s
    auto issue = [&](const ItemPos& ip, int slot, int L, int s) {
        const int h = ip.h, rb = ip.rb;
        const bool slot_ok = slot >= 0 && slot < p.num_slots;
        const bool len_ok = L >= 0 && L <= T;
        if (p.err != nullptr && h == 0 && rb == 0) {  // once per lane
            if (slot != -1 && !slot_ok)
                atomicOr(p.err, GDN_ERRBIT_INDEX);
            else if (slot_ok && !len_ok)
                atomicOr(p.err, GDN_ERRBIT_ACCEPT_LEN);
        }
        const bool active = slot_ok && len_ok && L > 0;
        st_slot[s] = active ? slot : -1;
        st_len[s] = L;
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
                tma_load_3d(base + s * CS::STAGE_BYTES + j * CS::BOX_BYTES, &tmap, j * CS::BOX_COLS, rb * ROWS,
                            slot * p.HV + h, bar);
        }
    };
    const int vj0 = warp * VPW + lane / LPV;  // this lane's vector in the first pass (before the j0 offset)
    const int vc = lane % LPV;                // its columns [8 vc, 8 vc + 8)
    const int j0 = kCommit ? T : 0;           // vectors j in [j0, 2T): q_j for j < T, k_{j-T} otherwise
    auto vec_ptr = [&](int b, int hk, int j) -> const InT* {
        const int t = j < T ? j : j - T;
        return static_cast<const InT*>(j < T ? p.q : p.k) + (((int64_t)b * T + t) * p.HK + hk) * DK + 8 * vc;
    };
    using IR = ItemRegs<DK, InT, kCommit>;
    auto load_regs = [&](const ItemPos& ip, bool need_qk, IR& r) {
#pragma unroll
        for (int ps = 0; ps < IR::NPASS; ++ps) {
            const int j = j0 + vj0 + ps * VPASS;
#pragma unroll
            for (int c = 0; c < QK::NC; ++c) r.raw[ps][c] = make_uint4(0, 0, 0, 0);
            if (need_qk && j < 2 * T) QK::load_global(vec_ptr(ip.b, ip.hk, j), r.raw[ps]);
        }
        const int row = ip.rb * ROWS + tid;
        const InT* vsrc = static_cast<const InT*>(p.v) + ((int64_t)ip.b * T * p.HV + ip.h) * p.DV + row;
#pragma unroll
        for (int t = 0; t < kChunkMaxT; ++t) {
            r.v[t] = InT(0.f);
            if (t < T && row < p.DV) r.v[t] = vsrc[(int64_t)t * p.HV * p.DV];
        }
        r.a = r.b = InT(0.f);
        r.A_log = r.dt_bias = 0.f;
        if (tid >= GATE_T0 && tid - GATE_T0 < T) {
            const int64_t ab = ((int64_t)ip.b * T + (tid - GATE_T0)) * p.HV + ip.h;
            r.a = static_cast<const InT*>(p.a)[ab];
            r.b = static_cast<const InT*>(p.b)[ab];
            r.A_log = p.A_log[ip.h];
            r.dt_bias = p.dt_bias[ip.h];
        }
    };

    ItemPos pos = ItemPos::of(beg, NRB, p.HV, R);  // the current item
    ItemPos ipos = pos;           // thread PT: the next item to issue, with its slot and token count
    int islot = 0, ilen = 0;
    if (tid == PT) {
        for (int s = 0; s < NS; ++s) mbar_init(ctl + 8 * s, 1);
        fence_mbar_init();
        islot = p.indices[ipos.b];
        ilen = kCommit ? p.steps[ipos.b] : T;
        for (int j = 0; j < NS - 1 && beg + j < end; ++j) {
            issue(ipos, islot, ilen, j);
            ipos.next(NRB, p.HV, R);
            if (beg + j + 1 < end) {
                islot = p.indices[ipos.b];
                ilen = kCommit ? p.steps[ipos.b] : T;
            }
        }
    }
    IR cur, nxt;
    load_regs(pos, true, cur);
    __syncthreads();

    uint32_t phase = 0;  // bit s: parity of the next completion of stage s
    int prev_b = -1, prev_hk = -1;
    for (int i = 0, it = beg; it < end; ++i, ++it) {
        const int st = i % NS;
        const int b = pos.b, h = pos.h, rb = pos.rb;
        const int hk = pos.hk;
        const int row0 = rb * ROWS;
        const int nrows = min(ROWS, p.DV - row0);
        const bool refill = it + NS - 1 < end;
        auto issue_ahead = [&] {  // thread PT: item it + NS - 1, then look up the slot of the one after it
            issue(ipos, islot, ilen, (i + NS - 1) % NS);
            ipos.next(NRB, p.HV, R);
            if (it + NS < end) {
                islot = p.indices[ipos.b];
                ilen = kCommit ? p.steps[ipos.b] : T;
            }
        };
        const int slot = st_slot[st];
        const int L = st_len[st];
        const bool active = slot >= 0;
        const bool reuse = b == prev_b && hk == prev_hk;  // same lane and key head: q, k, Gram still in place
        prev_b = b;
        prev_hk = hk;
        ItemPos npos = pos;
        npos.next(NRB, p.HV, R);
        if (it + 1 < end) load_regs(npos, !(npos.b == b && npos.hk == hk), nxt);

        if (active && !reuse) {
            // token prologue: normalise q and k into bf16 hi + lo rows of B
#pragma unroll
            for (int pass = 0; pass < IR::NPASS; ++pass) {
                if (j0 + pass * VPASS >= 2 * T) break;
                const int j = j0 + vj0 + pass * VPASS;
                float2 x[4];
                QK::unpack(cur.raw[pass], x);
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) ss = fmaf(x[e].x, x[e].x, fmaf(x[e].y, x[e].y, ss));
#pragma unroll
                for (int m = 1; m < LPV; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
                if (j < 2 * T) {
                    const float rn = rsqrtf(ss + p.l2_eps);
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        f[2 * e] = x[e].x * rn;
                        f[2 * e + 1] = x[e].y * rn;
                    }
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
                        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(f[2 * e] - __low2float(hi2),
                                                                         f[2 * e + 1] - __high2float(hi2));
                        hw[e] = *reinterpret_cast<const uint32_t*>(&hi2);
                        lw[e] = *reinterpret_cast<const uint32_t*>(&lo2);
                    }
                    const int t = j < T ? j : j - T;
                    const int hi_row = j < T ? 2 * T + t : t;  // q hi rows start at 2T, k hi rows at 0
                    *reinterpret_cast<uint4*>(Bs + hi_row * CS::ROW_BYTES + 16 * vc) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(Bs + (hi_row + T) * CS::ROW_BYTES + 16 * vc) =
                        make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            for (int i2 = CS::ncols(T) * (DK / 8) + tid; i2 < CS::b_rows(T) * (DK / 8); i2 += ROWS) {  // B padding
                const int r = i2 / (DK / 8), c = i2 - r * (DK / 8);
                *reinterpret_cast<uint4*>(Bs + r * CS::ROW_BYTES + 16 * c) = make_uint4(0, 0, 0, 0);
            }
        }
        __syncthreads();
        // the refill of the stage the last item used (the replay commit first waits for its store to have read
        // it) and the gates (needed only after the tile's wait) go in parallel with the Gram matrices
        if (refill && tid == PT) {
            if (kCommit) bulk_wait_read_all();
            issue_ahead();
        }
        if (active && tid >= GATE_T0 && tid - GATE_T0 < T) {
            gs[tid - GATE_T0] = gate(cur.A_log, to_f32(cur.a), cur.dt_bias);
            bs[tid - GATE_T0] = sigmoid(to_f32(cur.b));
        }

        if (active && !reuse && (warp == 1 || (!kCommit && warp == 0))) {
            // Gram matrices kh.kh (and kh.qh in verify mode) on the tensor cores, from the hi + lo rows of B:
            // A rows 0..7 address kh_0..kh_7 and rows 8..15 kl_0..kl_7, B columns 8 nb .. 8 nb + 7 address
            // block nb of B (kh, kl, qh, ql); rows past T point at row 0 and their products are dropped.  The
            // four products of a pair (hi.hi, hi.lo, lo.hi, lo.lo) then sit in one lane.  Warp 1 forms kh.kh from
            // blocks 0, 1; in verify, warp 0 forms kh.qh from blocks 2, 3 at the same time.
            constexpr int NB = 2;
            const int nb0 = warp == 1 ? 0 : 2;
            const int m = lane & 15;
            const int arow = m < 8 ? (m < T ? m : 0) : (m - 8 < T ? T + m - 8 : 0);
            const uint32_t a_addr = base + CS::b_off() + (uint32_t)arow * CS::ROW_BYTES + (lane >> 4) * 16;
            uint32_t b_addr[NB];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int jr = lane & 7;
                const int brow = jr < T ? (nb0 + nb) * T + jr : 0;
                b_addr[nb] = base + CS::b_off() + (uint32_t)brow * CS::ROW_BYTES + ((lane >> 3) & 1) * 16;
            }
            float g[NB][4];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int c = 0; c < 4; ++c) g[nb][c] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(a_addr + ks * 32, a0, a1, a2, a3);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    uint32_t b0, b1;
                    ldsm_x2(b_addr[nb] + ks * 32, b0, b1);
                    mma_bf16_16816(g[nb], a0, a1, a2, a3, b0, b1);
                }
            }
            const int s_ = lane >> 2;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t_ = 2 * (lane & 3) + e;
                if (s_ < T && t_ < T)
                    (warp == 1 ? KK : KQ)[t_ * TP + s_] = (g[0][e] + g[1][e]) + (g[0][2 + e] + g[1][2 + e]);
            }
        }
        // the state tile: bounded wait (uniform: every thread takes the same branch)
        bool ok = true;
        if (active) {
            ok = mbar_wait_bounded(ctl + 8 * st, (phase >> st) & 1u, kChunkWaitPolls);
            phase ^= 1u << st;
        }
        if (__syncthreads_or(!ok)) {
            if (tid == PT) {
                if (p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_TIMEOUT);
                // drain every tile still in flight (this one and the ones issued ahead) before leaving
                mbar_wait_bounded(ctl + 8 * st, ((phase >> st) & 1u) ^ 1u, kChunkWaitPolls);
                for (int j = 1; j < NS && it + j < end; ++j) {
                    const int s2 = (i + j) % NS;
                    if (st_slot[s2] >= 0) mbar_wait_bounded(ctl + 8 * s2, (phase >> s2) & 1u, kChunkWaitPolls);
                }
                if (kCommit) bulk_wait_all();
            }
            return;
        }

        if (active) {
            const uint32_t stage = base + st * CS::STAGE_BYTES;
            const int ra_row = warp * 32 + (lane & 15);  // the row this lane addresses in ldmatrix / stmatrix
            // this warp's P rows 0..15 and 16..31 (pbase[m] + r * p_stride, r < 16)
            float* pbase[2];
            {
                const int ps = CS::p_stride(T);
                unsigned char* own = sm + st * CS::STAGE_BYTES + warp * 32 * CS::SWZ;  // its rows in box 0
                float* Pw = kCommit              ? reinterpret_cast<float*>(sm + CS::p_off(T) + warp * CS::warp_region(T))
                            : CS::p_mode(T) <= 1 ? reinterpret_cast<float*>(own)
                            : CS::p_mode(T) == 2 ? reinterpret_cast<float*>(sm + st * CS::STAGE_BYTES) + warp * 32 * ps
                                                 : reinterpret_cast<float*>(sm + CS::p_off(T)) + warp * 32 * ps;
                pbase[0] = Pw;
                pbase[1] = CS::p_mode(T) == 1 ? reinterpret_cast<float*>(own + CS::BOX_BYTES) : Pw + 16 * ps;
            }
            // P = S_0 [kh hi | kh lo | qh hi | qh lo]^T on the tensor cores: warp w, rows [32w, 32w + 32)
            {
                const int NT8 = CS::b_rows(T) / 8;
                float acc[2][4][4];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[mt][nt][c] = 0.f;
                const int ra = ra_row;
                const uint32_t b_base =
                    base + CS::b_off() + (uint32_t)(lane & 7) * CS::ROW_BYTES + ((lane >> 3) & 1) * 16;
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    uint32_t a[2][4];
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
                        ldsm_x4(stage + swz_off<DK>(ra + mt * 16, 2 * ks + (lane >> 4)), a[mt][0], a[mt][1], a[mt][2],
                                a[mt][3]);
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        if (nt < NT8) {
                            uint32_t b0, b1;
                            ldsm_x2(b_base + nt * 8 * CS::ROW_BYTES + ks * 32, b0, b1);
#pragma unroll
                            for (int mt = 0; mt < 2; ++mt)
                                mma_bf16_16816(acc[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b0, b1);
                        }
                    }
                }
                if (CS::p_mode(T) == 2)
                    __syncthreads();  // every warp's A reads are done before P covers the stage
                else
                    __syncwarp();  // the warp's A reads are done before P covers its rows
                const int ps = CS::p_stride(T), ncol = CS::ncols(T);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int r = lane >> 2;  // row within the m tile; pbase[mt] holds the tile's first row
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        const int c = nt * 8 + (lane & 3) * 2;
                        if (nt < NT8) {
                            if (c < ncol) {
                                pbase[mt][r * ps + c] = acc[mt][nt][0];
                                pbase[mt][(r + 8) * ps + c] = acc[mt][nt][2];
                            }
                            if (c + 1 < ncol) {
                                pbase[mt][r * ps + c + 1] = acc[mt][nt][1];
                                pbase[mt][(r + 8) * ps + c + 1] = acc[mt][nt][3];
                            }
                        }
                    }
                }
            }
            __syncwarp();
            float* Pr = pbase[lane >> 4] + (lane & 15) * CS::p_stride(T);
            float vr[kChunkMaxT];
#pragma unroll
            for (int t = 0; t < kChunkMaxT; ++t) vr[t] = to_f32(cur.v[t]);

            if constexpr (kCommit) {
                // per row: the coefficients of the final state, as this warp's rows of A2
                unsigned char* a2w = sm + CS::p_off(T) + warp * CS::warp_region(T);
                switch (T) {
                case 1: row_coefficients<1>(Pr, vr, gs, bs, KK, L, a2w + lane * CS::a2_stride(T)); break;
                case 2: row_coefficients<2>(Pr, vr, gs, bs, KK, L, a2w + lane * CS::a2_stride(T)); break;
                case 3: row_coefficients<3>(Pr, vr, gs, bs, KK, L, a2w + lane * CS::a2_stride(T)); break;
                case 4: row_coefficients<4>(Pr, vr, gs, bs, KK, L, a2w + lane * CS::a2_stride(T)); break;
                case 5: row_coefficients<5>(Pr, vr, gs, bs, KK, L, a2w + lane * CS::a2_stride(T)); break;
                case 6: row_coefficients<6>(Pr, vr, gs, bs, KK, L, a2w + lane * CS::a2_stride(T)); break;
                case 7: row_coefficients<7>(Pr, vr, gs, bs, KK, L, a2w + lane * CS::a2_stride(T)); break;
                default: row_coefficients<8>(Pr, vr, gs, bs, KK, L, a2w + lane * CS::a2_stride(T)); break;
                }
                float gamma = 1.f;
                for (int t = 0; t < L; ++t) gamma *= gs[t];
                __syncwarp();
                // S_L = gamma S_0 + A2 [kh hi; kh hi; kh lo] on the tensor cores, 16 columns at a time: S_0 comes
                // in as the accumulator (ldmatrix gives the m16n8 accumulator layout of each 8 x 8 block) and
                // goes back over itself (stmatrix), each warp on its own rows
                const int KS2 = CS::a2_cols(T) / 16;
                const uint32_t a2b = base + CS::p_off(T) + warp * CS::warp_region(T) +
                                     (uint32_t)(lane & 15) * CS::a2_stride(T) + (lane >> 4) * 16;
                uint32_t af[2][2][4];  // [k step][m tile]
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
                        if (ks < KS2)
                            ldsm_x4(a2b + mt * 16 * CS::a2_stride(T) + ks * 32, af[ks][mt][0], af[ks][mt][1],
                                    af[ks][mt][2], af[ks][mt][3]);
                uint32_t brow[2];  // row of B2 (a row of B) that this lane addresses, per k step
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int kidx = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int r = kidx < T ? kidx : (kidx < 2 * T ? kidx - T : (kidx < 3 * T ? kidx - T : 0));
                    brow[ks] = base + CS::b_off() + (uint32_t)r * CS::ROW_BYTES + (lane >> 4) * 16;
                }
#pragma unroll 2
                for (int np = 0; np < DK / 16; ++np) {
                    float d[2][2][4];
                    uint32_t sa[2];
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        sa[mt] = stage + swz_off<DK>(ra_row + mt * 16, 2 * np + (lane >> 4));
                        uint32_t s0, s1, s2, s3;
                        ldsm_x4(sa[mt], s0, s1, s2, s3);
                        const float2 f0 = bf16x2_to_float2(s0), f1 = bf16x2_to_float2(s1);
                        const float2 f2 = bf16x2_to_float2(s2), f3 = bf16x2_to_float2(s3);
                        d[mt][0][0] = gamma * f0.x;
                        d[mt][0][1] = gamma * f0.y;
                        d[mt][0][2] = gamma * f1.x;
                        d[mt][0][3] = gamma * f1.y;
                        d[mt][1][0] = gamma * f2.x;
                        d[mt][1][1] = gamma * f2.y;
                        d[mt][1][2] = gamma * f3.x;
                        d[mt][1][3] = gamma * f3.y;
                    }
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        if (ks < KS2) {
                            uint32_t b00, b01, b10, b11;
                            ldsm_x4_trans(brow[ks] + np * 32, b00, b01, b10, b11);
#pragma unroll
                            for (int mt = 0; mt < 2; ++mt) {
                                mma_bf16_16816(d[mt][0], af[ks][mt][0], af[ks][mt][1], af[ks][mt][2], af[ks][mt][3], b00, b01);
                                mma_bf16_16816(d[mt][1], af[ks][mt][0], af[ks][mt][1], af[ks][mt][2], af[ks][mt][3], b10, b11);
                            }
                        }
                    }
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
                        stsm_x4(sa[mt], bf16x2_bits(d[mt][0][0], d[mt][0][1]), bf16x2_bits(d[mt][0][2], d[mt][0][3]),
                                bf16x2_bits(d[mt][1][0], d[mt][1][1]), bf16x2_bits(d[mt][1][2], d[mt][1][3]));
                }
                fence_proxy_async_smem();  // the stmatrix writes above, then the TMA store reads them
                __syncthreads();
                if (tid == PT) {
#pragma unroll
                    for (int j = 0; j < CS::NBOX; ++j)
                        tma_store_3d(&tmap, j * CS::BOX_COLS, row0, slot * p.HV + h, stage + j * CS::BOX_BYTES);
                    bulk_commit_group();
                }
            } else {
                // per row (one thread each, in the warp that computed it): the recurrence and the outputs
                const int r = warp * 32 + lane;
                const bool live = r < nrows;
                const int64_t o0 = ((int64_t)b * T * p.HV + h) * p.DV + row0 + r;
                const int64_t tok_out = (int64_t)p.HV * p.DV;
                switch (T) {
                case 1: row_recurrence<1>(p, Pr, vr, gs, bs, KK, KQ, live, o0, tok_out); break;
                case 2: row_recurrence<2>(p, Pr, vr, gs, bs, KK, KQ, live, o0, tok_out); break;
                case 3: row_recurrence<3>(p, Pr, vr, gs, bs, KK, KQ, live, o0, tok_out); break;
                case 4: row_recurrence<4>(p, Pr, vr, gs, bs, KK, KQ, live, o0, tok_out); break;
                case 5: row_recurrence<5>(p, Pr, vr, gs, bs, KK, KQ, live, o0, tok_out); break;
                case 6: row_recurrence<6>(p, Pr, vr, gs, bs, KK, KQ, live, o0, tok_out); break;
                case 7: row_recurrence<7>(p, Pr, vr, gs, bs, KK, KQ, live, o0, tok_out); break;
                default: row_recurrence<8>(p, Pr, vr, gs, bs, KK, KQ, live, o0, tok_out); break;
                }
                if (CS::p_mode(T) <= 2)
                    fence_proxy_async_smem();  // generic writes, then a TMA load refills the stage
            }
        }
        __syncthreads();  // the stage, B, P and the gates are free for the next item
        if (it + 1 < end) cur = nxt;
        pos = npos;
    }
    if (kCommit && tid == PT) bulk_wait_all();
}

// ---- host side ------------------------------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once (no link-time dependency on libcuda)
inline EncodeTiledFn encode_tiled_fn() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// The bf16 pool as a 3-D tensor [num_slots * HV][DV][DK]; box = (one swizzle span of columns, 128 rows, 1).
template <int DK>
cudaError_t encode_pool_map(CUtensorMap* map, void* pool, const RecurrentParams& p) {
    const EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    constexpr uint32_t SWZ = DK * 2 < 128 ? DK * 2 : 128;
    const cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)p.DV, (cuuint64_t)p.num_slots * (cuuint64_t)p.HV};
    const cuuint64_t strides[2] = {(cuuint64_t)DK * 2, (cuuint64_t)p.DV * DK * 2};
    const cuuint32_t box[3] = {SWZ / 2, (cuuint32_t)kChunkRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle sw =
        SWZ == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : (SWZ == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pool, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

constexpr int kChunkStages = 2;
constexpr int kChunkCachedDevices = 64;  // devices whose launch settings are cached

// grid = min(items, SMs x resident CTAs), each CTA a contiguous range of items
template <int DK, typename InT, bool kCommit>
cudaError_t launch_chunked(const RecurrentParams& p, int B, cudaStream_t s) {
    constexpr int NS = kChunkStages;
    using CS = ChunkPlan<DK, kCommit, NS>;
    auto kernel = gdn_verify_chunked_kernel<DK, InT, kCommit, NS>;
    const uint32_t smem = CS::bytes(p.T);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // Launch caches shared by every calling thread, one entry per device: the shared-memory opening is a
    // per-device attribute of the function, and occupancy may differ between devices.  A repeated first call
    // only repeats the same queries; devices beyond the table are queried on every call.
    static std::atomic<int> attr_bytes[kChunkCachedDevices];               // bytes opened on each device
    static std::atomic<int> occ_cache[kChunkCachedDevices][kChunkMaxT + 1];  // zero-initialised (static)
    const bool cached = dev >= 0 && dev < kChunkCachedDevices;
    if (!cached || (int)smem > attr_bytes[dev].load(std::memory_order_relaxed)) {
        const int most = (int)CS::bytes(kChunkMaxT);
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
        if (e != cudaSuccess) return e;
        if (cached) attr_bytes[dev].store(most, std::memory_order_relaxed);
    }
    int occ = cached ? occ_cache[dev][p.T].load(std::memory_order_relaxed) : 0;
    if (occ == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kChunkThreads, smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        if (cached) occ_cache[dev][p.T].store(occ, std::memory_order_relaxed);
    }
    CUtensorMap map;
    e = encode_pool_map<DK>(&map, kCommit ? p.pool_out : const_cast<void*>(p.pool_in), p);
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)B * p.HV * ((p.DV + kChunkRows - 1) / kChunkRows);
    if (items > INT32_MAX) return cudaErrorInvalidValue;
    const int64_t want = std::min<int64_t>(items, (int64_t)sms * occ);
    const int per_cta = (int)((items + want - 1) / want);
    const int grid = (int)((items + per_cta - 1) / per_cta);
    kernel<<<grid, kChunkThreads, smem, s>>>(p, map, (int)items, per_cta);
    return cudaGetLastError();
}

}  // namespace gdn
