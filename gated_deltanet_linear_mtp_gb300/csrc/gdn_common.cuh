// gdn_common.cuh -- device building blocks of the decode / verify kernels (sm_103a): storage conversions,
// 16-byte global accesses, the lane layout of a block of state rows, the per-token row update of the gated
// delta rule, the gate and beta scalars, and mbarrier / bulk-copy (TMA) wrappers.
//
// The rows of one state S[DV, DK] evolve independently:
//     u_i = (g s_i) . kh,   s_i <- g s_i + beta (v_i - u_i) kh,   o_i = s_i . qh
// so a CTA owns a block of rows of one (lane, value head) and keeps them in fp32 registers for all T tokens
// (layout: Split below).
//
// One sweep per token.  With a = s.kh and c = s.qh taken on the state before the token,
//     u = g a,  delta = beta (v_i - u),  s' = g s + delta kh,  o_i = g c + delta (kh . qh)
// which equals the plain order in exact arithmetic: both dot products come out of one pass over the
// registers, then one fused update.  kh . qh is formed once per token by the caller.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 16-byte state load, coherent, no L1 allocation (the state is read exactly once).
__device__ __forceinline__ uint4 ld_state16(const void* p) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte streaming store (evict-first): intermediate states are written once and not re-read here.
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_plain16(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Conversions between one 16-byte chunk and CH fp32 values.
template <typename StT>
struct Chunk;

template <>
struct Chunk<float> {
    static constexpr int CH = 4;
    __device__ __forceinline__ static void unpack(const uint4& r, float* s) {
        s[0] = __uint_as_float(r.x);
        s[1] = __uint_as_float(r.y);
        s[2] = __uint_as_float(r.z);
        s[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* s) {
        return make_uint4(__float_as_uint(s[0]), __float_as_uint(s[1]), __float_as_uint(s[2]), __float_as_uint(s[3]));
    }
};

template <>
struct Chunk<__nv_bfloat16> {
    static constexpr int CH = 8;
    __device__ __forceinline__ static void unpack(const uint4& r, float* s) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {  // element 2m sits in the low half (little endian)
            s[2 * m] = __uint_as_float(w[m] << 16);
            s[2 * m + 1] = __uint_as_float(w[m] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<const uint32_t*>(&v);
    }
    __device__ __forceinline__ static uint4 pack(const float* s) {
        return make_uint4(pack2(s[0], s[1]), pack2(s[2], s[3]), pack2(s[4], s[5]), pack2(s[6], s[7]));
    }
};

// Lane layout of one CTA's block of RPC state rows.  A row is split into P = DK / 8 slices of 8
// consecutive columns, one per lane; each lane holds the same slice of RL rows (RL = 4, or 2 when DK = 16),
// so the normalised k and q a lane needs for a token are only 8 columns of each.  A warp holds NRG = 32 / P
// row groups; lane (rg, p) of warp w owns rows w * RPW + i * NRG + rg (i < RL), columns [8p, 8p + 8).  A
// warp-wide access to "row i" of every row group thus covers NRG consecutive whole rows.
template <int DK>
struct Split {
    static constexpr int COLS = 8;
    static constexpr int P = DK / COLS;                     // lanes per row
    static constexpr int RL = P >= 4 ? 4 : P;               // rows per lane
    static constexpr int LOG_RL = RL == 4 ? 2 : (RL == 2 ? 1 : 0);
    static constexpr int NRG = 32 / P;                      // row groups per warp
    static constexpr int RPW = NRG * RL;                    // rows per warp
    // 4 warps per CTA: measured faster than 8-warp CTAs, whose prologue barrier idles more warps
    static constexpr int WARPS = 4;
    static constexpr int THREADS = 32 * WARPS;
    // resident CTAs an SM must fit (register cap, 80 a thread): 24 warps per SM hide the prologue's loads
    static constexpr int MIN_CTAS_PER_SM = 24 / WARPS;
    static constexpr int RPC = RPW * WARPS;                 // rows per CTA
    static_assert(P >= RL && 32 % P == 0, "DK must be 16, 32, 64, 128 or 256");

    // row (inside the CTA's block) of logical row slot j of lane (warp, rg)
    __device__ __forceinline__ static int row(int warp, int rg, int j) { return warp * RPW + j * NRG + rg; }
    // The logical row slot whose complete dot products lane p holds after the reduction in token_update.
    // A lane stores its rows in the order "register slot s holds logical slot s ^ own_slot(p)", so that at
    // every halving step of the reduction all lanes keep their first half and send their second half.
    __device__ __forceinline__ static int own_slot(int p) {
        int i = 0;
#pragma unroll
        for (int l = 0; l < LOG_RL; ++l)
            if (p & (P >> (l + 1))) i += RL >> (l + 1);
        return i;
    }
    // Shared-memory position of column `col` of a normalised k or q row.  Lane p reads its columns
    // [8p, 8p + 4) as one float4 at 4p and [8p + 4, 8p + 8) as one float4 at DK/2 + 4p, so the P lanes of a
    // row group read one contiguous, bank-conflict-free span per load.
    __host__ __device__ __forceinline__ static int kq_pos(int col) {
        return (col >> 3) * 4 + ((col & 4) ? DK / 2 : 0) + (col & 3);
    }
    // the lowest lane (p) holding the complete dot products of logical slot i
    __device__ __forceinline__ static int owner_p(int i) {
        int p = 0;
#pragma unroll
        for (int l = 0; l < LOG_RL; ++l)
            if (i & (RL >> (l + 1))) p += P >> (l + 1);
        return p;
    }
};

// 8 consecutive state elements (as 4 column pairs) <-> 16-byte chunks (1 for bf16, 2 for fp32)
template <typename StT>
struct Slice8 {
    static constexpr int NC = 8 / Chunk<StT>::CH;
    __device__ __forceinline__ static void unpack(const uint4 (&r)[NC], float2 (&s)[4]) {
        float f[8];
#pragma unroll
        for (int c = 0; c < NC; ++c) Chunk<StT>::unpack(r[c], f + c * Chunk<StT>::CH);
#pragma unroll
        for (int e = 0; e < 4; ++e) s[e] = make_float2(f[2 * e], f[2 * e + 1]);
    }
    __device__ __forceinline__ static void load_global(const StT* src, uint4 (&r)[NC]) {
#pragma unroll
        for (int c = 0; c < NC; ++c) r[c] = ld_state16(src + c * Chunk<StT>::CH);
    }
    __device__ __forceinline__ static void load_shared(const StT* src, float2 (&s)[4]) {
        uint4 r[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) r[c] = *reinterpret_cast<const uint4*>(src + c * Chunk<StT>::CH);
        unpack(r, s);
    }
    template <bool kStreaming>
    __device__ __forceinline__ static void store_global(StT* dst, const float2 (&s)[4]) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = s[e].x;
            f[2 * e + 1] = s[e].y;
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 v = Chunk<StT>::pack(f + c * Chunk<StT>::CH);
            if (kStreaming)
                st_stream16(dst + c * Chunk<StT>::CH, v);
            else
                st_plain16(dst + c * Chunk<StT>::CH, v);
        }
    }
};

// Per-lane constants of the token loop, computed once per CTA.
template <int DK>
struct LaneRows {
    using SP = Split<DK>;
    int code;               // own_slot(p): register slot s holds logical slot s ^ code
    int row[SP::RL];        // row (inside the CTA's block) held in register slot s
    int src[SP::RL];        // lane holding the delta of register slot s's row
    int own_row;            // row whose delta and output this lane forms
    __device__ __forceinline__ LaneRows(int warp, int rg, int p) {
        code = SP::own_slot(p);
#pragma unroll
        for (int s = 0; s < SP::RL; ++s) {
            row[s] = SP::row(warp, rg, s ^ code);
            src[s] = rg * SP::P + SP::owner_p(s ^ code);
        }
        own_row = SP::row(warp, rg, code);
    }
};

// One token on a lane's RL x 8 state elements, held as RL x 4 pairs of adjacent columns so that the dot
// products and the update run on packed fp32x2 multiply-adds (each half rounds like a scalar fmaf).
//   kt, qt   normalised k and q of the token (fp32, shared memory, DK each, columns at Split::kq_pos)
//   v_own    v of the token for the lane's own row (LaneRows::own_row)
// Row dot products a = s.kh and c = s.qh: 8-column partial sums (even and odd columns accumulate
// separately), then a transposed butterfly over the P lanes of the row group: at each of log2(RL) halving
// steps every lane keeps the first half of its rows and sends the second half to its partner (the
// lane-dependent register order of LaneRows makes the halves line up), then plain xor steps finish the
// sum.  Lane p ends with the complete sums of its own row, forms that row's delta and output, and the
// deltas of its RL rows are gathered back with shuffles for the update.  Returns the output (before
// scale) of the own row.
template <int DK>
__device__ __forceinline__ float token_update(float2 (&S)[Split<DK>::RL][4], const float* kt, const float* qt, float g,
                                              float beta, float v_own, float kq, int p, const LaneRows<DK>& lr) {
    using SP = Split<DK>;
    constexpr int RL = SP::RL;
    constexpr int P = SP::P;
    float2 k2[4], q2[4];
    {
        const float4 k0 = *reinterpret_cast<const float4*>(kt + 4 * p);
        const float4 k1 = *reinterpret_cast<const float4*>(kt + DK / 2 + 4 * p);
        const float4 q0 = *reinterpret_cast<const float4*>(qt + 4 * p);
        const float4 q1 = *reinterpret_cast<const float4*>(qt + DK / 2 + 4 * p);
        k2[0] = make_float2(k0.x, k0.y);
        k2[1] = make_float2(k0.z, k0.w);
        k2[2] = make_float2(k1.x, k1.y);
        k2[3] = make_float2(k1.z, k1.w);
        q2[0] = make_float2(q0.x, q0.y);
        q2[1] = make_float2(q0.z, q0.w);
        q2[2] = make_float2(q1.x, q1.y);
        q2[3] = make_float2(q1.z, q1.w);
    }
    float a[RL], c[RL];
#pragma unroll
    for (int i = 0; i < RL; ++i) {
        float2 ak = make_float2(0.f, 0.f), cq = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ak = __ffma2_rn(S[i][e], k2[e], ak);
            cq = __ffma2_rn(S[i][e], q2[e], cq);
        }
        a[i] = ak.x + ak.y;
        c[i] = cq.x + cq.y;
    }
#pragma unroll
    for (int l = 0; l < SP::LOG_RL; ++l) {
        const int m = P >> (l + 1);
#pragma unroll
        for (int j = 0; j < (RL >> (l + 1)); ++j) {
            a[j] += __shfl_xor_sync(0xffffffffu, a[j + (RL >> (l + 1))], m);
            c[j] += __shfl_xor_sync(0xffffffffu, c[j + (RL >> (l + 1))], m);
        }
    }
#pragma unroll
    for (int m = P >> (SP::LOG_RL + 1); m >= 1; m >>= 1) {
        a[0] += __shfl_xor_sync(0xffffffffu, a[0], m);
        c[0] += __shfl_xor_sync(0xffffffffu, c[0], m);
    }
    const float delta = beta * (v_own - g * a[0]);
    const float out = fmaf(g, c[0], delta * kq);
    const float2 g2 = make_float2(g, g);
#pragma unroll
    for (int i = 0; i < RL; ++i) {
        const float d = __shfl_sync(0xffffffffu, delta, lr.src[i]);
        const float2 d2 = make_float2(d, d);
#pragma unroll
        for (int e = 0; e < 4; ++e) S[i][e] = __ffma2_rn(d2, k2[e], __fmul2_rn(g2, S[i][e]));
    }
    return out;
}

// g = exp(-exp(A_log) * softplus(a + dt_bias)),  softplus(x) = log(1 + e^x) (written x + log(1 + e^-x) for x > 0)
__device__ __forceinline__ float gate(float A_log, float a, float dt_bias) {
    const float x = a + dt_bias;
    const float sp = x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
    return expf(-expf(A_log) * sp);
}

__device__ __forceinline__ float sigmoid(float x) { return 1.f / (1.f + expf(-x)); }

// ---- mbarrier and bulk-copy (TMA) wrappers ----------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the phase with the given parity: false if it did not complete within `limit` polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Global -> shared bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned), completing on
// the mbarrier `bar` of this CTA.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Polls of one mbarrier wait before the wait is declared failed (the kernel then sets GDN_ERRBIT_TIMEOUT and
// leaves the work it waited for undone).  A test build lowers it, together with GDN_TEST_MISSING_COPY, which
// leaves one copy unissued so that its wait runs out (tests/test_gpu_timeout.py).
#ifndef GDN_WAIT_POLLS
#define GDN_WAIT_POLLS (1u << 22)
#endif

// Position of a work item of the persistent kernels: items are numbered row block fastest, then value head,
// then lane, and a CTA walks a contiguous range of them without dividing.
struct ItemPos {
    int b, h, rb;  // lane, value head, row block
    int hk, hr;    // key head h / R and h % R, R = value heads per key head
    __device__ __forceinline__ static ItemPos of(int it, int NRB, int HV, int R) {
        ItemPos q;
        q.rb = it % NRB;
        const int bh = it / NRB;
        q.h = bh % HV;
        q.b = bh / HV;
        q.hk = q.h / R;
        q.hr = q.h - q.hk * R;
        return q;
    }
    __device__ __forceinline__ void next(int NRB, int HV, int R) {
        if (++rb == NRB) {
            rb = 0;
            if (++hr == R) {
                hr = 0;
                ++hk;
            }
            if (++h == HV) {
                h = hk = hr = 0;
                ++b;
            }
        }
    }
};

}  // namespace gdn
