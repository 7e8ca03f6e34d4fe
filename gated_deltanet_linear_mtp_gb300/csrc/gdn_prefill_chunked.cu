// gdn_prefill_chunked.cu -- prefill in chunked form on the tensor cores (sm_103a, tcgen05 with the state held in
// tensor memory), for DK in {64, 128}.  The call's definition is the one of gdn_prefill.cu: sequence b owns tokens
// cu_seqlens[b] .. cu_seqlens[b+1]-1, starts from its pool slot (or from zero when has_initial_state[b] == 0),
// writes o at every token and its final state back into the slot.  The chunked gated delta rule with bf16 state
// pools and the initial-state mask of TensorRT-LLM PR #20937 (Per-File QA Perspective, Source files and
// Test-code files: the chunked prefill kernel and its fresh-state zeroing).
//
// Chunked form.  Within a chunk of C = 32 tokens t = 0 .. C-1 starting from state S_0, with
// gamma_t = g_0 ... g_t, G(s,t) = g_{s+1} ... g_t (G(t,t) = 1) and delta_t = beta_t (v_t - g_t S_{t-1} kh_t),
// the recurrence unrolls to (the same algebra as the chunked verify):
//     u_t   = g_t S_{t-1} kh_t = gamma_t (S_0 kh_t) + sum_{s<t}  G(s,t) (kh_s . kh_t) delta_s,   delta_t = beta_t (v_t - u_t)
//     o_t   = scale S_t qh_t   = scale (gamma_t (S_0 qh_t) + sum_{s<=t} G(s,t) (kh_s . qh_t) delta_s)
//     S_C-1 = gamma_{C-1} S_0 + sum_s G(s, C-1) delta_s kh_s^T .
// The dense work is on the tensor cores in bf16 operands with fp32 accumulation, each fp32 operand split into
// hi = bf16(x) and lo = bf16(x - hi) (about 16 significant bits; the lo.lo part products, about 2^-18 relative,
// are left out):
//   Gram   of the chunk's k and q rows (M = 128, N = C or 2C; A and B from shared memory),
//   P      S_0 [k; q]^T (M = 128 state rows; A = S_0 hi / lo written into tensor memory),
//   O      delta KQw^T, onto gamma_t S_0 qh_t (A = delta hi / lo in tensor memory, B = KQw hi / lo),
//   update S += c k (N = DK; A = c_s = G(s, C-1) delta_s hi / lo in tensor memory, B = the k rows read MN-major),
//          onto gamma_{C-1} S_0 written in place beforehand;
// what is left per state row is the u recurrence above, in fp32 registers, one thread per row.  The state stays
// in fp32 in tensor memory for the whole sequence and is rounded to the pool's type once, at the final write-back,
// like the token loop's registers.
//
// Two ways to bring the tokens in.  bf16 q, k, v (with v in whole 16-byte pieces and DV >= 128) arrive by TMA:
// raw k and q rows straight into the swizzled operand buffer (a bf16 value is its own hi part, its lo part is
// zero) and v as a bf16 tile; the L2 normalisation is then a factor per token, rk_t = 1 / sqrt(|k_t|^2 + eps)
// (and rq_t), with |k_t|^2 and |q_t|^2 read off the diagonal of the Gram product [k; q][k; q]^T, applied to P in
// the row thread, to the weights, and to the update's coefficients.  Otherwise (fp32 inputs, odd layouts) the
// token group loads and normalises q and k itself into [kh hi | qh hi | kh lo | qh lo] rows and stores v as fp32.
//
// CTA = one item = (sequence, value head, block of 128 state rows); a kernel that allocates tensor memory runs one
// CTA per SM.  Warps 0-3 (the row group, thread = state row = tensor-memory lane) run the state chain: S_0 into
// hi / lo, the P product, the row recurrence, the O and update products, o out.  Warps 4-7 (the token group)
// prepare the next chunk meanwhile in a ring of buffer stages: the token rows, v, the gates with their prefix and
// suffix products, the Gram product and from it the decay-weighted matrices KKw[t][s] = G(s,t) kh_s . kh_t (s < t)
// and KQw[t][s] = G(s,t) kh_s . qh_t (s <= t).  mbarriers hand the stages back and forth (every wait bounded: a
// wait that runs out sets GDN_ERRBIT_TIMEOUT and the CTA leaves).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tcgen05.cuh"

#include <atomic>
#include <cstring>
#include <type_traits>

namespace gdn {
namespace {

constexpr int kPC = 32;          // tokens per chunk
constexpr int kPRows = 128;      // state rows per item: the MMA's M, the tensor-memory lanes
constexpr int kPThreads = 256;   // the row group (warps 0-3) and the token group (warps 4-7)
constexpr int kBarRow = 1, kBarTok = 2;  // named barriers of the two groups (0 is the CTA's)
constexpr uint32_t kPWaitPolls = GDN_WAIT_POLLS;
constexpr uint32_t kPCols = 512;  // tensor memory of the CTA (a power of two covering the plan)

template <int DK, bool kTma>
struct PrefillChunkPlan {
    static_assert(DK == 64 || DK == 128, "the chunked prefill takes DK = 64 or 128");
    static constexpr int NST = kTma ? 3 : 2;  // buffer stages (TMA: one chunk of lead for the loads)
    // stacked token rows per 64-column box: [k | q] raw bf16 (TMA), or [kh hi | qh hi | kh lo | qh lo]
    static constexpr int KQR = kTma ? 2 * kPC : 4 * kPC;
    static constexpr uint32_t BOX = KQR * 128u;
    static constexpr uint32_t KQ_BYTES = BOX * (DK / 64);
    // TMA: the Gram product's A spans 128 rows, 64 past the stacked ones, which must still be shared memory
    static constexpr uint32_t KQ_PAD = kTma ? 64u * 128u : 0u;
    // KQw in bf16 hi then lo, the B operand of the O product: C rows of 128 bytes each (K = C of 64 columns used)
    static constexpr uint32_t KQB_BYTES = 2u * kPC * 128u;
    static constexpr uint32_t KQB_OFF = NST * KQ_BYTES + KQ_PAD;
    static constexpr uint32_t VT_BYTES = kTma ? kPC * kPRows * 2u : 0u;  // TMA: v as bf16 [token][128 rows]
    static constexpr uint32_t VT_OFF = KQB_OFF + NST * KQB_BYTES;
    // floats of a stage: KKwT [s][t]; v [token][row] (no TMA); per token g, beta, gamma, the update's factor
    // G(s, C-1) rk_s, the P factors gamma_t rk_t and gamma_t rq_t, rk, rq (rk = rq = 1 when normalised beforehand)
    static constexpr int KKW = 0, VB = kPC * kPC, GG = VB + (kTma ? 0 : kPC * kPRows), BET = GG + kPC,
                         GAM = BET + kPC, CEND = GAM + kPC, GK = CEND + kPC, GQ = GK + kPC, RK = GQ + kPC,
                         RQ = RK + kPC, F_FLOATS = RQ + kPC;
    static constexpr uint32_t F_OFF = VT_OFF + NST * VT_BYTES;
    static constexpr int SCR_STRIDE = kPC + 1;  // partial Gram rows (no TMA), padded against bank conflicts
    static constexpr uint32_t SCR_OFF = F_OFF + NST * F_FLOATS * 4u;
    // two chunks of o staged for the stores: [token][128 rows] in o's type (fp32 at most)
    static constexpr uint32_t OB_BYTES = kPC * kPRows * 4u;
    static constexpr uint32_t OB_OFF = (SCR_OFF + 64u * SCR_STRIDE * 4u + 1023u) & ~1023u;
    static constexpr uint32_t BAR_OFF = OB_OFF + 2u * OB_BYTES;
    static constexpr uint32_t BYTES = BAR_OFF + 256u + 1024u;  // + the alignment slack of the base
    static_assert(KQB_OFF % 1024 == 0 && VT_OFF % 1024 == 0 && F_OFF % 16 == 0, "operand alignment");
    // tensor-memory columns: S (fp32), S_0 hi and lo (bf16 pairs; delta hi and lo after the P product), P, the Gram
    // product (two of C columns, or one of 2C), c hi and lo, O
    static constexpr uint32_t S_COL = 0, SH_COL = DK, SL_COL = DK + DK / 2, P_COL = 2 * DK, G1_COL = P_COL + 4 * kPC,
                              G2_COL = G1_COL + kPC, CH_COL = G2_COL + kPC, CL_COL = CH_COL + kPC / 2,
                              O_COL = CL_COL + kPC / 2, COLS = O_COL + kPC;
    static_assert(COLS <= kPCols, "tensor memory of the plan");
};

// mbarriers, 8 bytes each from the plan's BAR_OFF: per stage full (token group -> row group), empty (the update
// product that read the stage has completed) and TMA (the stage's token rows have landed)
enum {
    kFull0 = 0, kEmpty0 = 3, kTmaBar0 = 6, kPBar = 9, kUpdBar, kGramBar, kDrainRow, kDrainTok, kNumBars
};

template <typename T>
__device__ __forceinline__ void load16(const T* src, float (&f)[16]);
template <>
__device__ __forceinline__ void load16<__nv_bfloat16>(const __nv_bfloat16* src, float (&f)[16]) {
    const uint4 a = reinterpret_cast<const uint4*>(src)[0], b = reinterpret_cast<const uint4*>(src)[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float2 x = bf16x2_to_float2(w[e]);
        f[2 * e] = x.x;
        f[2 * e + 1] = x.y;
    }
}
template <>
__device__ __forceinline__ void load16<float>(const float* src, float (&f)[16]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float4 x = reinterpret_cast<const float4*>(src)[e];
        f[4 * e] = x.x;
        f[4 * e + 1] = x.y;
        f[4 * e + 2] = x.z;
        f[4 * e + 3] = x.w;
    }
}

template <typename T>
__device__ __forceinline__ void store16(T* dst, const float (&f)[16]);
template <>
__device__ __forceinline__ void store16<__nv_bfloat16>(__nv_bfloat16* dst, const float (&f)[16]) {
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = bf16x2_bits(f[2 * e], f[2 * e + 1]);
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
}
template <>
__device__ __forceinline__ void store16<float>(float* dst, const float (&f)[16]) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
        reinterpret_cast<float4*>(dst)[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
}

// x = hi + lo in bf16 pairs (element 2e in the low half): hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
    hi = *reinterpret_cast<const uint32_t*>(&h2);
    lo = bf16x2_bits(x0 - __low2float(h2), x1 - __high2float(h2));
}

template <int DK, typename InT, typename StT, bool kTma>
__global__ void __launch_bounds__(kPThreads, 1)
    gdn_prefill_chunked_kernel(const RecurrentParams p, const int32_t* __restrict__ cu_seqlens,
                               const int32_t* __restrict__ has_init, int n_tokens,
                               const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap kmap,
                               const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap vmap,
                               int o_tma) {
    using PL = PrefillChunkPlan<DK, kTma>;
    constexpr int C = kPC;
    constexpr int NST = PL::NST;
    const int NRB = (p.DV + kPRows - 1) / kPRows;
    const int item = blockIdx.x;  // row block fastest, then value head, then sequence
    const int rb = item % NRB, h = (item / NRB) % p.HV, b = item / (NRB * p.HV);
    const int hk = h / (p.HV / p.HK);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int lt = tid & (kPRows - 1);  // index in the group = tensor-memory lane
    const bool row_group = tid < kPRows;
    const int row = rb * kPRows + lt;   // row group: the state row; token group: the row of v it loads

    // lane gather, then the sequence's bounds, checked like the token loop (index first)
    const int slot = p.indices[b];
    const bool reporter = p.err != nullptr && tid == 0 && rb == 0 && h == 0;  // once per sequence
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
    const int nch = (n + C - 1) / C;

    extern __shared__ unsigned char pc_smem[];
    const uint32_t raw_base = smem_u32(pc_smem);
    const uint32_t pad = ((raw_base + 1023u) & ~1023u) - raw_base;
    unsigned char* sm = pc_smem + pad;
    const uint32_t base = raw_base + pad;
    const uint32_t bars = base + PL::BAR_OFF;
    auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
    volatile int* fail = reinterpret_cast<volatile int*>(sm + PL::BAR_OFF + 8 * kNumBars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + PL::BAR_OFF + 8 * kNumBars + 8);
    float* scr = reinterpret_cast<float*>(sm + PL::SCR_OFF);

    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kPCols);
    if (tid == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(bar(kFull0 + i), kPRows);
        for (int i = kEmpty0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        *fail = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    auto fbuf = [&](int st) -> float* { return reinterpret_cast<float*>(sm + PL::F_OFF) + st * PL::F_FLOATS; };
    auto kq_addr = [&](int st) -> uint32_t { return base + (uint32_t)st * PL::KQ_BYTES; };
    auto kqb_addr = [&](int st) -> uint32_t { return base + PL::KQB_OFF + (uint32_t)st * PL::KQB_BYTES; };
    auto vtile = [&](int st) -> const __nv_bfloat16* {
        return reinterpret_cast<const __nv_bfloat16*>(sm + PL::VT_OFF + (size_t)st * PL::VT_BYTES);
    };

    if (row_group) {
        // ================================ row group: the state chain ================================
        const bool live = row < p.DV;
        bool issued = false;  // thread 0: an MMA was issued (drained before leaving)
        // initial state: the pool row in fp32 tensor memory, zero for a fresh sequence
        {
            const StT* src = static_cast<const StT*>(p.pool_in) + (((int64_t)slot * p.HV + h) * p.DV + row) * DK;
#pragma unroll
            for (int c0 = 0; c0 < DK; c0 += 16) {
                float f[16];
                if (live && !fresh) {
                    load16<StT>(src + c0, f);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) f[e] = 0.f;
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(f[e]);
                tmem_st8(lane_base + PL::S_COL + c0, w);
                tmem_st8(lane_base + PL::S_COL + c0 + 8, w + 8);
            }
            tmem_wait_st();
        }
        // o: o_t = scale O_t, O = gamma_t S_0 qh_t + sum_s KQw[t][s] delta_s formed on the tensor cores in its own
        // columns (read back in the next chunk while its P product runs); staged in shared memory and written by one
        // TMA tensor store per whole chunk (o as [tokens][HV][DV], box 32 x 1 x 128), or by bulk copies of the
        // block's rows per token, or, when o allows neither, stored directly
        const uint32_t osz = p.out_bf16 ? 2u : 4u;
        const bool o_bulk = (reinterpret_cast<uintptr_t>(p.o) & 15u) == 0 && ((int64_t)p.DV * osz) % 16 == 0;
        const uint32_t blk_bytes = (uint32_t)min(kPRows, p.DV - rb * kPRows) * osz;
        const int64_t tok_out = (int64_t)p.HV * p.DV;
        auto emit_o = [&](int cc) {
            if (o_bulk) {  // 16 tokens at a time, not unrolled (less code beside the other warp group's)
                unsigned char* ob = sm + PL::OB_OFF + (cc & 1) * PL::OB_BYTES;
#pragma unroll 1
                for (int t0 = 0; t0 < C; t0 += 16) {
                    float oh[16];
                    tmem_ld16(lane_base + PL::O_COL + t0, oh);
                    tmem_wait_ld();
                    if (p.out_bf16) {
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            reinterpret_cast<__nv_bfloat16*>(ob)[(t0 + t) * kPRows + lt] =
                                __float2bfloat16_rn(p.scale * oh[t]);
                    } else {
#pragma unroll
                        for (int t = 0; t < 16; ++t) reinterpret_cast<float*>(ob)[(t0 + t) * kPRows + lt] = p.scale * oh[t];
                    }
                }
                fence_proxy_async_smem();  // read by the bulk copies
                return;
            }
            float ov[C];
            tmem_ld16(lane_base + PL::O_COL, ov);
            tmem_ld16(lane_base + PL::O_COL + 16, ov + 16);
            tmem_wait_ld();
            if (live) {
                const int len = min(C, n - cc * C);
                const int64_t o0 = ((int64_t)(lo + cc * C) * p.HV + h) * p.DV + row;
                if (p.out_bf16) {
#pragma unroll
                    for (int t = 0; t < C; ++t)
                        if (t < len)
                            static_cast<__nv_bfloat16*>(p.o)[o0 + t * tok_out] = __float2bfloat16_rn(p.scale * ov[t]);
                } else {
#pragma unroll
                    for (int t = 0; t < C; ++t)
                        if (t < len) static_cast<float*>(p.o)[o0 + t * tok_out] = p.scale * ov[t];
                }
            }
        };
        constexpr int kOT = 96;  // the thread that issues and waits for the o copies (not the MMA issuer)
        auto issue_o = [&](int cc) {  // thread kOT, after a barrier behind every row's emit_o(cc)
            const int len = min(C, n - cc * C);
            const uint32_t ob = base + PL::OB_OFF + (uint32_t)(cc & 1) * PL::OB_BYTES;
            if (o_tma && len == C) {
                tma_store_3d(&omap, rb * kPRows, h, lo + cc * C, ob);
            } else {  // the sequence's last, partial chunk: the box would run into the next sequence
                for (int t = 0; t < len; ++t)
                    bulk_s2g(static_cast<unsigned char*>(p.o) +
                                 (((int64_t)(lo + cc * C + t) * p.HV + h) * p.DV + rb * kPRows) * osz,
                             ob + (uint32_t)t * kPRows * osz, blk_bytes);
            }
            bulk_commit_group();
        };
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int st = c % NST;
            const float* F = fbuf(st);
            const uint32_t kq = kq_addr(st);
            bool w = mbar_wait_bounded(bar(kFull0 + st), (uint32_t)(c / NST) & 1u, kPWaitPolls);
            if (w && c > 0) w = mbar_wait_bounded(bar(kUpdBar), (uint32_t)(c - 1) & 1u, kPWaitPolls);
            // the staging buffer of chunk c-1's o was last copied from for chunk c-3, two groups ago
            if (lt == kOT && o_bulk && c >= 3) bulk_wait_read_but_one();
            if (named_sync_or(kBarRow, kPRows, !w || *fail != 0)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // S_0 -> bf16 hi / lo (the A operand of P), and gamma_{C-1} S_0 back in place for the update, 32 columns
            // at a time with the next block's load in flight
            const float gend = F[PL::GAM + C - 1];
            {
                float f[2][32];
                tmem_ld16(lane_base + PL::S_COL, f[0]);
                tmem_ld16(lane_base + PL::S_COL + 16, f[0] + 16);
                tmem_wait_ld();
                // a loop over pairs of blocks, not unrolled: the two warp groups' code shares each scheduler's
                // instruction cache, and instruction fetch was the leading stall (measured 4% faster)
#pragma unroll 1
                for (int jp = 0; jp < DK / 32; jp += 2)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int jb = jp + jj;
                    const int c0 = 32 * jb;
                    float(&x)[32] = f[jj];
                    if (jb + 1 < DK / 32) {
                        tmem_ld16(lane_base + PL::S_COL + c0 + 32, f[jj ^ 1]);
                        tmem_ld16(lane_base + PL::S_COL + c0 + 48, f[jj ^ 1] + 16);
                    }
                    uint32_t hw[16], lw[16], sw[32];
                    const float2 g2 = make_float2(gend, gend), m1 = make_float2(-1.f, -1.f);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float2 x2 = make_float2(x[2 * e], x[2 * e + 1]);
                        const __nv_bfloat162 h2 = __float22bfloat162_rn(x2);
                        hw[e] = *reinterpret_cast<const uint32_t*>(&h2);
                        const float2 r2 = __ffma2_rn(bf16x2_to_float2(hw[e]), m1, x2);  // x - hi, exact
                        lw[e] = bf16x2_bits(r2.x, r2.y);
                        const float2 s2 = __fmul2_rn(g2, x2);
                        sw[2 * e] = __float_as_uint(s2.x);
                        sw[2 * e + 1] = __float_as_uint(s2.y);
                    }
                    tmem_st8(lane_base + PL::SH_COL + c0 / 2, hw);
                    tmem_st8(lane_base + PL::SH_COL + c0 / 2 + 8, hw + 8);
                    tmem_st8(lane_base + PL::SL_COL + c0 / 2, lw);
                    tmem_st8(lane_base + PL::SL_COL + c0 / 2 + 8, lw + 8);
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmem_st8(lane_base + PL::S_COL + c0 + 8 * q, sw + 8 * q);
                    if (jb + 1 < DK / 32) tmem_wait_ld();
                }
            }
            tmem_wait_st();
            tc_fence_before();
            named_sync(kBarRow, kPRows);
            // P = S_0 [stacked rows]^T: S_0 hi against every stacked row, S_0 lo against the hi rows (TMA: the raw
            // k and q rows, N = 2C; otherwise [kh hi | qh hi | kh lo | qh lo], N = 4C and 2C)
            if (lt == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    const uint64_t bd = umma_desc_sw128(kq + (uint32_t)(ks >> 2) * PL::BOX + (uint32_t)(ks & 3) * 32u);
                    umma_bf16_ta(tmem + PL::P_COL, tmem + PL::SH_COL + 8 * ks, bd,
                                 umma_idesc_bf16(kPRows, kTma ? 2 * C : 4 * C), ks > 0 ? 1u : 0u);
                    umma_bf16_ta(tmem + PL::P_COL, tmem + PL::SL_COL + 8 * ks, bd, umma_idesc_bf16(kPRows, 2 * C), 1u);
                }
                umma_commit(bar(kPBar));
                issued = true;
            }
            if (c > 0) emit_o(c - 1);  // while the P product runs
            const bool pw = mbar_wait_bounded(bar(kPBar), (uint32_t)c & 1u, kPWaitPolls);
            if (named_sync_or(kBarRow, kPRows, !pw)) {
                ok = false;
                break;
            }
            if (lt == kOT && c > 0 && o_bulk) issue_o(c - 1);
            tc_fence_after();
            // this row of P: S_0 k_t = P[t] (+ P[2C + t]), S_0 q_t = P[C + t] (+ P[3C + t])
            float pk[C], pq[C];
            {
                tmem_ld16(lane_base + PL::P_COL, pk);
                tmem_ld16(lane_base + PL::P_COL + 16, pk + 16);
                tmem_ld16(lane_base + PL::P_COL + C, pq);
                tmem_ld16(lane_base + PL::P_COL + C + 16, pq + 16);
                tmem_wait_ld();
                if constexpr (!kTma) {
                    float x[C];
                    tmem_ld16(lane_base + PL::P_COL + 2 * C, x);
                    tmem_ld16(lane_base + PL::P_COL + 2 * C + 16, x + 16);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < C; ++t) pk[t] += x[t];
                    tmem_ld16(lane_base + PL::P_COL + 3 * C, x);
                    tmem_ld16(lane_base + PL::P_COL + 3 * C + 16, x + 16);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < C; ++t) pq[t] += x[t];
                }
            }
            // the row's u recurrence, right-looking: once delta_s is known it goes into u_t of every later token
            // (KKwT[s][t] = KKw[t][s], zero for t <= s), so the dependent chain per token is a few operations and
            // the rest are independent FMAs
            const float* KKwT = F + PL::KKW;
            uint32_t ow[C];  // gamma_t S_0 qh_t, the O product's starting value
#pragma unroll
            for (int t = 0; t < C; ++t) {
                pk[t] *= F[PL::GK + t];  // gamma_t rk_t: gamma_t S_0 kh_t
                ow[t] = __float_as_uint(F[PL::GQ + t] * pq[t]);
            }
            uint32_t dhw[C / 2], dlw[C / 2], chw[C / 2], clw[C / 2];
            float dprev = 0.f, cprev = 0.f;
            const __nv_bfloat16* vt = vtile(st);
#pragma unroll
            for (int s = 0; s < C; ++s) {
                const float vs = kTma ? __bfloat162float(vt[s * kPRows + lt]) : F[PL::VB + s * kPRows + lt];
                const float ds = F[PL::BET + s] * (vs - pk[s]);
#pragma unroll
                for (int t4 = (s + 1) & ~3; t4 < C; t4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(KKwT + s * C + t4);
                    if (t4 > s) pk[t4] = fmaf(a4.x, ds, pk[t4]);
                    if (t4 + 1 > s) pk[t4 + 1] = fmaf(a4.y, ds, pk[t4 + 1]);
                    if (t4 + 2 > s) pk[t4 + 2] = fmaf(a4.z, ds, pk[t4 + 2]);
                    if (t4 + 3 > s) pk[t4 + 3] = fmaf(a4.w, ds, pk[t4 + 3]);
                }
                // delta_s (the O product's A) and c_s = G(s, C-1) rk_s delta_s (the update's A) in hi / lo pairs
                const float cs = F[PL::CEND + s] * ds;
                if (s & 1) {
                    split_pair(dprev, ds, dhw[s / 2], dlw[s / 2]);
                    split_pair(cprev, cs, chw[s / 2], clw[s / 2]);
                } else {
                    dprev = ds;
                    cprev = cs;
                }
            }
#pragma unroll
            for (int jj = 0; jj < C / 2; jj += 8) {
                tmem_st8(lane_base + PL::SH_COL + jj, dhw + jj);
                tmem_st8(lane_base + PL::SL_COL + jj, dlw + jj);
                tmem_st8(lane_base + PL::CH_COL + jj, chw + jj);
                tmem_st8(lane_base + PL::CL_COL + jj, clw + jj);
            }
#pragma unroll
            for (int jj = 0; jj < C; jj += 8) tmem_st8(lane_base + PL::O_COL + jj, ow + jj);
            tmem_wait_st();
            tc_fence_before();
            named_sync(kBarRow, kPRows);  // every row's operands are in place; every read of stage st is done
            if (lt == 0) {
                tc_fence_after();
                // O += (delta hi + delta lo)(KQw hi + KQw lo)^T without the lo.lo part: B = the C rows of KQw, K-major
                const uint32_t kqb = kqb_addr(st);
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int bh = 0; bh < 2 - a; ++bh)
#pragma unroll
                        for (int ks = 0; ks < C / 16; ++ks)
                            umma_bf16_ta(tmem + PL::O_COL, tmem + (a ? PL::SL_COL : PL::SH_COL) + 8 * ks,
                                         umma_desc_sw128(kqb + (uint32_t)bh * (C * 128u) + 32u * ks),
                                         umma_idesc_bf16(kPRows, C), 1u);
                // S += (c hi + c lo) k: B = the k rows read MN-major (TMA: raw rows 0..C-1; otherwise kh hi rows
                // 0..C-1 against c hi and lo, and kh lo rows 2C..3C-1 against c hi)
                const uint32_t idesc = umma_idesc_bf16(kPRows, DK) | (1u << 16);
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int bh = 0; bh < (kTma ? 1 : 2 - a); ++bh)
#pragma unroll
                        for (int ks = 0; ks < C / 16; ++ks) {
                            const uint32_t brow = (uint32_t)(bh * 2 * C + 16 * ks);
                            umma_bf16_ta(tmem + PL::S_COL, tmem + (a ? PL::CL_COL : PL::CH_COL) + 8 * ks,
                                         umma_desc_sw128_mn(kq + brow * 128u, PL::BOX), idesc, 1u);
                        }
                umma_commit(bar(kUpdBar));  // also tracks the O product issued before it
                umma_commit(bar(kEmpty0 + st));  // the token group may refill stage st
            }
        }
        if (ok) {  // the last chunk's o, and the final state into the slot, rounded to the pool's type
            const bool uw = mbar_wait_bounded(bar(kUpdBar), (uint32_t)(nch - 1) & 1u, kPWaitPolls);
            if (lt == kOT && o_bulk && nch >= 3) bulk_wait_read_but_one();
            if (named_sync_or(kBarRow, kPRows, !uw)) {
                ok = false;
            } else {
                tc_fence_after();
                emit_o(nch - 1);
                StT* dst = static_cast<StT*>(p.pool_out) + (((int64_t)slot * p.HV + h) * p.DV + row) * DK;
#pragma unroll
                for (int c0 = 0; c0 < DK; c0 += 16) {
                    float f[16];
                    tmem_ld16(lane_base + PL::S_COL + c0, f);
                    tmem_wait_ld();
                    if (live) store16<StT>(dst + c0, f);
                }
                named_sync(kBarRow, kPRows);
                if (lt == kOT && o_bulk) issue_o(nch - 1);
            }
        }
        if (lt == kOT && o_bulk) bulk_wait_all();  // the o copies are complete before the CTA leaves
        if (!ok && lt == 0) {
            *fail = 1;
            if (p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_TIMEOUT);
        }
        if (lt == 0 && issued) {  // every MMA of this group has completed before the tensor memory is released
            umma_commit(bar(kDrainRow));
            mbar_wait_bounded(bar(kDrainRow), 0u, kPWaitPolls);
        }
    } else if constexpr (kTma) {
        // ================= token group (TMA): raw k, q rows into the operand stage, v as a bf16 tile =================
        const float A_log = p.A_log[h], dt_bias = p.dt_bias[h];
        const __nv_bfloat16* ap = static_cast<const __nv_bfloat16*>(p.a);
        const __nv_bfloat16* bp = static_cast<const __nv_bfloat16*>(p.b);
        __nv_bfloat16 araw = __float2bfloat16_rn(0.f), braw = araw;
        auto load_ab = [&](int cc) {  // lane = token of chunk cc
            if (lt < C && cc * C + lt < n) {
                araw = ap[(int64_t)(lo + cc * C + lt) * p.HV + h];
                braw = bp[(int64_t)(lo + cc * C + lt) * p.HV + h];
            }
        };
        constexpr uint32_t kTmaBytes = (2u * DK * C + (uint32_t)C * kPRows) * 2u;  // k, q boxes and the v box
        int tma_issued = 0;  // thread 0: chunks whose loads have been issued
        auto issue_tma = [&](int cc) {
            const int sg = cc % NST;
            const uint32_t tb = bar(kTmaBar0 + sg), kqs = kq_addr(sg);
            tma_issued = cc + 1;
#ifdef GDN_TEST_MISSING_COPY
            // test build: the first chunk of the first item is never loaded nor arrived on: its wait runs out
            if (item == 0 && cc == 0) return;
#endif
            mbar_arrive_expect_tx(tb, kTmaBytes);
#pragma unroll
            for (int j = 0; j < DK / 64; ++j) {
                tma_load_3d(kqs + (uint32_t)j * PL::BOX, &kmap, 64 * j, hk, lo + cc * C, tb);
                tma_load_3d(kqs + (uint32_t)j * PL::BOX + C * 128u, &qmap, 64 * j, hk, lo + cc * C, tb);
            }
            tma_load_3d(base + PL::VT_OFF + (uint32_t)sg * PL::VT_BYTES, &vmap, rb * kPRows, h, lo + cc * C, tb);
        };
        if (lt == 0) {
            issue_tma(0);
            if (nch > 1) issue_tma(1);
        }
        load_ab(0);
        bool issued = false, ok = true;
        int consumed = 0;
        for (int c = 0; c < nch; ++c) {
            const int st = c % NST;
            float* F = fbuf(st);
            const uint32_t kq = kq_addr(st);
            const bool w = mbar_wait_bounded(bar(kTmaBar0 + st), (uint32_t)(c / NST) & 1u, kPWaitPolls);
            if (named_sync_or(kBarTok, kPRows, !w || *fail != 0)) {
                ok = w;
                break;
            }
            consumed = c + 1;
            const int len = min(C, n - c * C);
            if (len < C) {  // the rows past the sequence hold another sequence's tokens (or zeros): clear them
                unsigned char* KQ = sm + (size_t)st * PL::KQ_BYTES;
                for (int i = lt; i < (C - len) * (DK / 8); i += kPRows) {
                    const int r = len + i / (DK / 8), c8 = i % (DK / 8);
                    *reinterpret_cast<uint4*>(KQ + sw128(PL::KQR, r, c8)) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(KQ + sw128(PL::KQR, C + r, c8)) = make_uint4(0, 0, 0, 0);
                }
                unsigned char* VT = sm + PL::VT_OFF + (size_t)st * PL::VT_BYTES;
                for (int i = lt; i < (C - len) * (kPRows / 8); i += kPRows)
                    *reinterpret_cast<uint4*>(VT + (size_t)(len + i / (kPRows / 8)) * kPRows * 2 + (i % (kPRows / 8)) * 16) =
                        make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();  // the cleared rows are read by the tensor cores
            }
            // gates (lane = token), with gamma_t = g_0 .. g_t and G(s, C-1) = g_{s+1} .. g_{C-1}
            float ce = 1.f;
            if (lt < C) {
                const bool valid = lt < len;  // tokens past the sequence: g = 1, beta = 0
                const float g = valid ? gate(A_log, __bfloat162float(araw), dt_bias) : 1.f;
                const float be = valid ? sigmoid(__bfloat162float(braw)) : 0.f;
                float gm = g, sf = g;
#pragma unroll
                for (int m = 1; m < 32; m <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gm, m);
                    if (lt >= m) gm *= y;
                    const float z = __shfl_down_sync(0xffffffffu, sf, m);
                    if (lt + m < 32) sf *= z;
                }
                ce = __shfl_down_sync(0xffffffffu, sf, 1);
                if (lt == C - 1) ce = 1.f;
                F[PL::GG + lt] = g;
                F[PL::BET + lt] = be;
                F[PL::GAM + lt] = gm;
            }
            named_sync(kBarTok, kPRows);
            // Gram product [k; q] [k; q]^T of the raw rows (rows 2C.. of A lie past the stage: their lanes are unused)
            if (lt == 0) {
                tc_fence_after();
                const uint32_t idesc = umma_idesc_bf16(kPRows, 2 * C);
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    const uint32_t koff = (uint32_t)(ks >> 2) * PL::BOX + (uint32_t)(ks & 3) * 32u;
                    umma_bf16(tmem + PL::G1_COL, umma_desc_sw128(kq + koff), umma_desc_sw128(kq + koff), idesc,
                              ks > 0 ? 1u : 0u);
                }
                umma_commit(bar(kGramBar));
                issued = true;
            }
            if (c + 1 < nch) load_ab(c + 1);  // in flight meanwhile
            const bool gw = mbar_wait_bounded(bar(kGramBar), (uint32_t)c & 1u, kPWaitPolls);
            if (named_sync_or(kBarTok, kPRows, !gw)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // lane t: k_t . [k; q], lane C + t: q_t . [k; q]; the diagonal gives |k_t|^2 and |q_t|^2
            float d[2 * C];
            if (lt < 2 * C) {
#pragma unroll
                for (int j = 0; j < 2 * C; j += 16) tmem_ld16(lane_base + PL::G1_COL + j, d + j);
                tmem_wait_ld();
                float nrm = 0.f;
#pragma unroll
                for (int j = 0; j < C; ++j) {
                    const float x = lt < C ? d[j] : d[C + j];
                    if (j == (lt & (C - 1))) nrm = x;
                }
                const int t = lt & (C - 1);
                F[(lt < C ? PL::RK : PL::RQ) + t] = t < len ? rsqrtf(nrm + p.l2_eps) : 0.f;
            }
            tc_fence_before();
            named_sync(kBarTok, kPRows);
            if (lt < 2 * C) {
                const int t = lt & (C - 1);
                const bool isq = lt >= C;  // rows C..2C-1: q_t . k_s
                const float rt = F[(isq ? PL::RQ : PL::RK) + t];
                float wv[C];
                float G = 1.f;  // G(s, t), built downwards from s = t
#pragma unroll
                for (int s = C - 1; s >= 0; --s) {
                    if (s < t) G *= F[PL::GG + s + 1];
                    wv[s] = (isq ? s <= t : s < t) ? G * (F[PL::RK + s] * rt) * d[s] : 0.f;
                }
                if (isq) {  // row t of KQw in bf16 hi / lo, K-major rows of 128 bytes (the O product's B)
                    unsigned char* kb = sm + PL::KQB_OFF + (size_t)st * PL::KQB_BYTES;
#pragma unroll
                    for (int j8 = 0; j8 < C / 8; ++j8) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) split_pair(wv[8 * j8 + 2 * e], wv[8 * j8 + 2 * e + 1], hw[e], lw[e]);
                        *reinterpret_cast<uint4*>(kb + sw128(C, t, j8)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(kb + C * 128 + sw128(C, t, j8)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                    fence_proxy_async_smem();
                } else {  // column t of KKwT (fp32, for the row recurrence), and the token's factors
                    float* dst = F + PL::KKW + t;
#pragma unroll
                    for (int s = 0; s < C; ++s) dst[s * C] = wv[s];
                    const float gm = F[PL::GAM + t];
                    F[PL::GK + t] = gm * rt;
                    F[PL::GQ + t] = gm * F[PL::RQ + t];
                    F[PL::CEND + t] = ce * rt;
                }
            }
            mbar_arrive(bar(kFull0 + st));  // after this thread's writes of the chunk
            // the loads of chunk c + 2, into the stage of chunk c - 1 once its update product has completed
            if (lt == 0 && c + 2 < nch) {
                const bool e = c < 1 || mbar_wait_bounded(bar(kEmpty0 + (c + 2) % NST),
                                                          (uint32_t)((c - 1) / NST) & 1u, kPWaitPolls);
                if (e)
                    issue_tma(c + 2);
                else
                    *fail = 1;
            }
        }
        if ((!ok || *fail != 0) && lt == 0) {
            *fail = 1;
            if (p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_TIMEOUT);
        }
        if (lt == 0) {  // loads issued and not consumed land, and every MMA completes, before the CTA leaves
            for (int cc = consumed; cc < tma_issued; ++cc)
                mbar_wait_bounded(bar(kTmaBar0 + cc % NST), (uint32_t)(cc / NST) & 1u, kPWaitPolls);
            if (issued) {
                umma_commit(bar(kDrainTok));
                mbar_wait_bounded(bar(kDrainTok), 0u, kPWaitPolls);
            }
        }
    } else {
        // ========== token group (no TMA): q, k loaded and normalised into hi / lo rows, v stored as fp32 ==========
        using QK = Slice8<InT>;
        constexpr int LPV = DK / 8;          // threads per q or k vector, 8 columns each
        constexpr int VPP = kPRows / LPV;    // vectors per pass of the group
        constexpr int NPASS = 2 * C / VPP;   // k_0 .. k_{C-1}, q_0 .. q_{C-1}
        const int vj0 = lt / LPV, vc = lt % LPV;
        const float A_log = p.A_log[h], dt_bias = p.dt_bias[h];
        const InT* qp = static_cast<const InT*>(p.q);
        const InT* kp = static_cast<const InT*>(p.k);
        const InT* vp = static_cast<const InT*>(p.v);
        const InT* ap = static_cast<const InT*>(p.a);
        const InT* bp = static_cast<const InT*>(p.b);
        uint4 raw[NPASS][QK::NC];
        constexpr int VPASS = C * kPRows / 8 / kPRows;  // 8-row pieces of v per thread and chunk
        uint4 vraw[VPASS][QK::NC];
        const int vrow = 8 * (lt % 16), vtok = lt / 16;  // this thread's v piece: rows vrow.., token vtok + 8 pass
        const int vrows = min(8, p.DV - (row - lt) - vrow);  // rows of the piece inside DV (<= 0: none)
        InT araw = InT(0.f), braw = InT(0.f);
        auto load_chunk = [&](int c) {
            const int t0 = c * C;
#pragma unroll
            for (int ps = 0; ps < NPASS; ++ps) {
                const int j = vj0 + ps * VPP;
                const int t = j < C ? j : j - C;
#pragma unroll
                for (int e = 0; e < QK::NC; ++e) raw[ps][e] = make_uint4(0, 0, 0, 0);
                if (t0 + t < n)
                    QK::load_global((j < C ? kp : qp) + ((int64_t)(lo + t0 + t) * p.HK + hk) * DK + 8 * vc, raw[ps]);
            }
#pragma unroll
            for (int ps = 0; ps < VPASS; ++ps) {
                const int t = vtok + 8 * ps;
#pragma unroll
                for (int e = 0; e < QK::NC; ++e) vraw[ps][e] = make_uint4(0, 0, 0, 0);
                if (t0 + t < n && vrows > 0) {
                    const InT* src = vp + ((int64_t)(lo + t0 + t) * p.HV + h) * p.DV + (row - lt) + vrow;
                    if (p.v_vec && vrows == 8) {
                        QK::load_global(src, vraw[ps]);
                    } else {  // a piece across the end of DV, or v not in 16-byte pieces
                        InT* dst = reinterpret_cast<InT*>(vraw[ps]);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (e < vrows) dst[e] = src[e];
                    }
                }
            }
            if (lt < C && t0 + lt < n) {
                araw = ap[(int64_t)(lo + t0 + lt) * p.HV + h];
                braw = bp[(int64_t)(lo + t0 + lt) * p.HV + h];
            }
        };
        bool issued = false;
        bool ok = true;
        load_chunk(0);
        for (int c = 0; c < nch; ++c) {
            const int st = c % NST;
            float* F = fbuf(st);
            unsigned char* KQ = sm + (size_t)st * PL::KQ_BYTES;
            const uint32_t kq = kq_addr(st);
            // stage st is free once the update of chunk c - NST (which read it last) has completed
            const bool w =
                c < NST || mbar_wait_bounded(bar(kEmpty0 + st), (uint32_t)((c - NST) / NST) & 1u, kPWaitPolls);
            if (named_sync_or(kBarTok, kPRows, !w || *fail != 0)) {
                ok = w;
                break;
            }
            // gates (lane = token of the chunk), with gamma_t = g_0 .. g_t and G(s, C-1) = g_{s+1} .. g_{C-1}
            if (lt < C) {
                const bool valid = c * C + lt < n;  // tokens past the sequence: g = 1, beta = 0, zero q and k
                const float g = valid ? gate(A_log, to_f32(araw), dt_bias) : 1.f;
                const float be = valid ? sigmoid(to_f32(braw)) : 0.f;
                float gm = g, sf = g;
#pragma unroll
                for (int m = 1; m < 32; m <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gm, m);
                    if (lt >= m) gm *= y;
                    const float z = __shfl_down_sync(0xffffffffu, sf, m);
                    if (lt + m < 32) sf *= z;
                }
                float ce = __shfl_down_sync(0xffffffffu, sf, 1);
                if (lt == C - 1) ce = 1.f;
                F[PL::GG + lt] = g;
                F[PL::BET + lt] = be;
                F[PL::GAM + lt] = gm;
                F[PL::CEND + lt] = ce;  // q and k are normalised here: the factors rk = rq = 1
                F[PL::GK + lt] = gm;
                F[PL::GQ + lt] = gm;
            }
            // v of the block's rows, per token
#pragma unroll
            for (int ps = 0; ps < VPASS; ++ps) {
                float2 x[4];
                QK::unpack(vraw[ps], x);
                float4* dst = reinterpret_cast<float4*>(F + PL::VB + (vtok + 8 * ps) * kPRows + vrow);
                dst[0] = make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
                dst[1] = make_float4(x[2].x, x[2].y, x[3].x, x[3].y);
            }
            // q, k normalised, into the stacked rows: kh hi at t, qh hi at C + t, kh lo at 2C + t, qh lo at 3C + t
#pragma unroll
            for (int ps = 0; ps < NPASS; ++ps) {
                const int j = vj0 + ps * VPP;
                float2 x[4];
                QK::unpack(raw[ps], x);
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) ss = fmaf(x[e].x, x[e].x, fmaf(x[e].y, x[e].y, ss));
#pragma unroll
                for (int m = 1; m < LPV; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
                const int t = j < C ? j : j - C;
                const float rn = c * C + t < n ? rsqrtf(ss + p.l2_eps) : 0.f;  // rows past the sequence: zero
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split_pair(x[e].x * rn, x[e].y * rn, hw[e], lw[e]);
                const int hrow = j;  // k_t: row t; q_t: row C + t (j = C + t)
                *reinterpret_cast<uint4*>(KQ + sw128(PL::KQR, hrow, vc)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(KQ + sw128(PL::KQR, hrow + 2 * C, vc)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            fence_proxy_async_smem();  // the rows are read by the tensor cores
            named_sync(kBarTok, kPRows);
            // Gram products [kh; qh] kh hi^T and [kh; qh] kh lo^T over all four parts of the stacked rows
            if (lt == 0) {
                tc_fence_after();
                const uint32_t idesc = umma_idesc_bf16(kPRows, C);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < DK / 16; ++ks) {
                        const uint32_t koff = (uint32_t)(ks >> 2) * PL::BOX + (uint32_t)(ks & 3) * 32u;
                        umma_bf16(tmem + (part ? PL::G2_COL : PL::G1_COL), umma_desc_sw128(kq + koff),
                                  umma_desc_sw128(kq + (uint32_t)(part * 2 * C) * 128u + koff), idesc,
                                  ks > 0 ? 1u : 0u);
                    }
                umma_commit(bar(kGramBar));
                issued = true;
            }
            if (c + 1 < nch) load_chunk(c + 1);  // in flight meanwhile
            const bool gw = mbar_wait_bounded(bar(kGramBar), (uint32_t)c & 1u, kPWaitPolls);
            if (named_sync_or(kBarTok, kPRows, !gw)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // lane m of the products holds stacked row m against kh_s: rows 2C.. (the lo parts) hand their sums
            // to rows 0..2C-1 through shared memory
            float gr[C];
            {
                float x[C];
                tmem_ld16(lane_base + PL::G1_COL, gr);
                tmem_ld16(lane_base + PL::G1_COL + 16, gr + 16);
                tmem_ld16(lane_base + PL::G2_COL, x);
                tmem_ld16(lane_base + PL::G2_COL + 16, x + 16);
                tmem_wait_ld();
#pragma unroll
                for (int s = 0; s < C; ++s) gr[s] += x[s];
            }
            if (lt >= 2 * C) {
#pragma unroll
                for (int s = 0; s < C; ++s) scr[(lt - 2 * C) * PL::SCR_STRIDE + s] = gr[s];
            }
            tc_fence_before();
            named_sync(kBarTok, kPRows);
            if (lt < 2 * C) {
                const int t = lt & (C - 1);
                const bool isq = lt >= C;  // rows C..2C-1: qh_t . kh_s
                float wv[C];
                float G = 1.f;  // G(s, t), built downwards from s = t
#pragma unroll
                for (int s = C - 1; s >= 0; --s) {
                    if (s < t) G *= F[PL::GG + s + 1];
                    const float full = gr[s] + scr[lt * PL::SCR_STRIDE + s];
                    wv[s] = (isq ? s <= t : s < t) ? G * full : 0.f;
                }
                if (isq) {  // row t of KQw in bf16 hi / lo, K-major rows of 128 bytes (the O product's B)
                    unsigned char* kb = sm + PL::KQB_OFF + (size_t)st * PL::KQB_BYTES;
#pragma unroll
                    for (int j8 = 0; j8 < C / 8; ++j8) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) split_pair(wv[8 * j8 + 2 * e], wv[8 * j8 + 2 * e + 1], hw[e], lw[e]);
                        *reinterpret_cast<uint4*>(kb + sw128(C, t, j8)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(kb + C * 128 + sw128(C, t, j8)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                    fence_proxy_async_smem();
                } else {  // column t of KKwT (fp32, for the row recurrence)
                    float* dst = F + PL::KKW + t;
#pragma unroll
                    for (int s = 0; s < C; ++s) dst[s * C] = wv[s];
                }
            }
            mbar_arrive(bar(kFull0 + st));  // after this thread's writes of the chunk
        }
        if (!ok && lt == 0) {
            *fail = 1;
            if (p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_TIMEOUT);
        }
        if (lt == 0 && issued) {
            umma_commit(bar(kDrainTok));
            mbar_wait_bounded(bar(kDrainTok), 0u, kPWaitPolls);
        }
    }
    // every tensor-memory access of both groups is complete before the allocation is released
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kPCols);
}

// A token-major tensor [n_tokens][heads][cols] (bf16 or fp32) as a 3-D tensor map with box (bx, 1, kPC): bx columns
// of one head for a chunk of tokens; the 128-byte swizzle for operand rows of 64 bf16, none otherwise.  False when
// the driver's encoder is missing or refuses the layout.
bool encode_tokens_map(CUtensorMap* map, const void* ptr, bool bf16, int cols, int heads, int n_tokens, int bx,
                       bool swizzle128) {
    const EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return false;
    const cuuint64_t esz = bf16 ? 2 : 4;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)n_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * esz, (cuuint64_t)heads * cols * esz};
    const cuuint32_t box[3] = {(cuuint32_t)bx, 1, (cuuint32_t)kPC};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TokenMaps {
    CUtensorMap o, k, q, v;
    int o_tma;
};

template <int DK, typename InT, typename StT, bool kTma>
cudaError_t launch_variant(const RecurrentParams& p, const int32_t* cu_seqlens, const int32_t* has_init, int B,
                           int n_tokens, const TokenMaps& m, cudaStream_t s) {
    using PL = PrefillChunkPlan<DK, kTma>;
    auto kernel = gdn_prefill_chunked_kernel<DK, InT, StT, kTma>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // the shared-memory attribute is per device: set once for each
    static std::atomic<uint64_t> ready{0};
    if (dev >= 64 || !(ready.load(std::memory_order_acquire) >> dev & 1u)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PL::BYTES);
        if (e != cudaSuccess) return e;
        if (dev < 64) ready.fetch_or(1ull << dev, std::memory_order_acq_rel);
    }
    const int NRB = (p.DV + kPRows - 1) / kPRows;
    const int64_t items = (int64_t)B * p.HV * NRB;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    kernel<<<(unsigned)items, kPThreads, PL::BYTES, s>>>(p, cu_seqlens, has_init, n_tokens, m.o, m.k, m.q, m.v,
                                                         m.o_tma);
    return cudaGetLastError();
}

template <int DK, typename InT, typename StT>
cudaError_t launch_dk(const RecurrentParams& p, const int32_t* cu_seqlens, const int32_t* has_init, int B,
                      int n_tokens, cudaStream_t s) {
    TokenMaps m;
    std::memset(&m, 0, sizeof m);
    // o: one TMA store per whole chunk when o is in 16-byte pieces and DV >= 128 (else per-token copies or stores)
    const uint64_t osz = p.out_bf16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(p.o) & 15u) == 0 && ((uint64_t)p.DV * osz) % 16 == 0 && p.DV >= kPRows &&
        n_tokens > 0)
        m.o_tma = encode_tokens_map(&m.o, p.o, p.out_bf16 != 0, p.DV, p.HV, n_tokens, kPRows, false);
    // bf16 q, k, v: the loads by TMA (q and k are 16-byte aligned by the interface's rules)
    if constexpr (std::is_same<InT, __nv_bfloat16>::value) {
        if (p.v_vec && p.DV >= kPRows && n_tokens > 0 &&
            encode_tokens_map(&m.k, p.k, true, DK, p.HK, n_tokens, 64, true) &&
            encode_tokens_map(&m.q, p.q, true, DK, p.HK, n_tokens, 64, true) &&
            encode_tokens_map(&m.v, p.v, true, p.DV, p.HV, n_tokens, kPRows, false))
            return launch_variant<DK, InT, StT, true>(p, cu_seqlens, has_init, B, n_tokens, m, s);
    }
    return launch_variant<DK, InT, StT, false>(p, cu_seqlens, has_init, B, n_tokens, m, s);
}

template <typename InT, typename StT>
cudaError_t launch_t(const RecurrentParams& p, const int32_t* cu, const int32_t* init, int B, int N, int DK,
                     cudaStream_t s) {
    switch (DK) {
    case 64: return launch_dk<64, InT, StT>(p, cu, init, B, N, s);
    case 128: return launch_dk<128, InT, StT>(p, cu, init, B, N, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool prefill_chunked_eligible(int DK) { return DK == 64 || DK == 128; }

cudaError_t launch_prefill_chunked(const RecurrentParams& p, const int32_t* cu_seqlens, const int32_t* has_init, int B,
                                   int n_tokens, int DK, bool qkv_bf16, bool state_bf16, cudaStream_t s) {
    if (state_bf16)
        return qkv_bf16 ? launch_t<__nv_bfloat16, __nv_bfloat16>(p, cu_seqlens, has_init, B, n_tokens, DK, s)
                        : launch_t<float, __nv_bfloat16>(p, cu_seqlens, has_init, B, n_tokens, DK, s);
    return qkv_bf16 ? launch_t<__nv_bfloat16, float>(p, cu_seqlens, has_init, B, n_tokens, DK, s)
                    : launch_t<float, float>(p, cu_seqlens, has_init, B, n_tokens, DK, s);
}

}  // namespace gdn
