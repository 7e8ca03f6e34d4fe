// gdn_gated_norm.cu -- gated RMSNorm of the recurrence's outputs (sm_103a):
//     y[r, i] = o[r, i] / sqrt(mean_i(o[r, i]^2) + eps) * w[i] * silu(z[r, i]),   silu(x) = x * sigmoid(x)
// for every row r of DV outputs (one value head of one token).  The decode-rows gated norm of TensorRT-LLM
// PR #20937 (GB300 Qwen3.8-Flash-Next NVFP4), Per-File QA Perspective, Source files; the page names the
// fusion, the formula is the plain reading (RMS over DV, one weight per column, gate after the norm).
//
// HBM-bound: o and z are read once, y written once (w stays in L1/L2).  GS consecutive lanes share a row;
// each lane takes 8 consecutive columns at a time (16-byte loads for bf16, two for fp32).  Rows of up to
// 1024 columns (NCH <= 4 chunks a lane): the lane loads its o and z chunks together into registers, the
// group reduces the sum of squares with shuffles, and y is formed from the registers -- one round trip to
// memory per row.  Wider rows loop over their chunks and re-read them (L1 hits) for y; a row that is not a
// multiple of 8 columns or not 16-byte aligned takes that loop one column at a time.  Every element is
// read and written by the same thread, so y may be o itself.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn_internal.h"

namespace gdn {

namespace {

__device__ __forceinline__ float ld1(const float* p) { return *p; }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st1(float* p, float x) { *p = x; }
__device__ __forceinline__ void st1(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// 8 consecutive elements <-> fp32
__device__ __forceinline__ void ld8(const float* p, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float (&f)[8]) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {  // element 2m sits in the low half
        f[2 * m] = __uint_as_float(w[m] << 16);
        f[2 * m + 1] = __uint_as_float(w[m] & 0xffff0000u);
    }
}
__device__ __forceinline__ void st8(float* p, const float (&f)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(f[2 * m], f[2 * m + 1]);
        w[m] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// silu on CUDA's fast exponential and division intrinsics: a few ulp of fp32 (about 1e-6 relative for the gates'
// range), far inside the norm's tolerance, and the limits hold (x -> -inf: e^-x overflows, the quotient is 0).  With
// the IEEE forms the kernel was bound by issue, not by HBM (344 against 283 us per launch at 2M rows of 128).
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

constexpr int kNormThreads = 256;

// Rows of at most 8 * GS * NCH columns (DV % 8 == 0, 16-byte aligned): everything from registers.  The weights
// are loaded with o and z, before the reduction (loaded after it, their latency sat between the reduction and
// the stores: 281.7 against 276.8 us per launch at 2M rows of 128).
// A row of a padded or invalid lane (when the call names the lanes' slots): left untouched.
__device__ __forceinline__ bool skipped_row(const GatedNormParams& q, int64_t row) {
    if (q.lane_slot == nullptr) return false;
    const int s = q.lane_slot[row / q.rows_per_lane];
    return s < 0 || s >= q.num_slots;
}

template <typename OT, typename ZT, int GS, int NCH>
__global__ void __launch_bounds__(kNormThreads) gdn_gated_rmsnorm_reg_kernel(const OT* o, const ZT* z, const float* w,
                                                                             OT* y, int64_t rows, int DV, float eps,
                                                                             const GatedNormParams q) {
    const int64_t row = ((int64_t)blockIdx.x * kNormThreads + threadIdx.x) / GS;
    const int gl = threadIdx.x % GS;
    if (row >= rows || skipped_row(q, row)) return;  // whole groups leave together: a group shares its row
    const unsigned mask = GS == 32 ? 0xffffffffu : (((1u << GS) - 1u) << ((threadIdx.x & 31) & ~(GS - 1)));
    const OT* orow = o + row * DV;
    const ZT* zrow = z + row * DV;
    float f[NCH][8], g[NCH][8], wv[NCH][8];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
        const int c = 8 * (gl + j * GS);
        if (c < DV) {
            ld8(orow + c, f[j]);
            ld8(zrow + c, g[j]);
            ld8(w + c, wv[j]);
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NCH; ++j)
        if (8 * (gl + j * GS) < DV)
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(f[j][e], f[j][e], ss);
#pragma unroll
    for (int m = GS / 2; m >= 1; m >>= 1) ss += __shfl_xor_sync(mask, ss, m);
    const float inv_rms = 1.f / sqrtf(ss / (float)DV + eps);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
        const int c = 8 * (gl + j * GS);
        if (c < DV) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[j][e] = f[j][e] * inv_rms * wv[j][e] * silu(g[j][e]);
            st8(y + row * DV + c, f[j]);
        }
    }
}

// Any row: a loop over 8-column chunks (kVec) or single columns, re-reading o for y.
template <typename OT, typename ZT, int GS, bool kVec>
__global__ void __launch_bounds__(kNormThreads) gdn_gated_rmsnorm_kernel(const OT* o, const ZT* z, const float* w,
                                                                         OT* y, int64_t rows, int DV, float eps,
                                                                         const GatedNormParams q) {
    const int64_t row = ((int64_t)blockIdx.x * kNormThreads + threadIdx.x) / GS;
    const int gl = threadIdx.x % GS;
    if (row >= rows || skipped_row(q, row)) return;  // whole groups leave together: a group shares its row
    const unsigned mask = GS == 32 ? 0xffffffffu : (((1u << GS) - 1u) << ((threadIdx.x & 31) & ~(GS - 1)));
    const OT* orow = o + row * DV;
    const ZT* zrow = z + row * DV;
    OT* yrow = y + row * DV;
    float ss = 0.f;
    if (kVec) {
        for (int c = 8 * gl; c < DV; c += 8 * GS) {
            float f[8];
            ld8(orow + c, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
        }
    } else {
        for (int i = gl; i < DV; i += GS) {
            const float f = ld1(orow + i);
            ss = fmaf(f, f, ss);
        }
    }
#pragma unroll
    for (int m = GS / 2; m >= 1; m >>= 1) ss += __shfl_xor_sync(mask, ss, m);
    const float inv_rms = 1.f / sqrtf(ss / (float)DV + eps);
    if (kVec) {
        for (int c = 8 * gl; c < DV; c += 8 * GS) {
            float f[8], g[8], wv[8];
            ld8(orow + c, f);
            ld8(zrow + c, g);
            ld8(w + c, wv);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = f[e] * inv_rms * wv[e] * silu(g[e]);
            st8(yrow + c, f);
        }
    } else {
        for (int i = gl; i < DV; i += GS) st1(yrow + i, ld1(orow + i) * inv_rms * w[i] * silu(ld1(zrow + i)));
    }
}

template <typename OT, typename ZT, int GS, bool kVec>
cudaError_t launch_norm_gs(const GatedNormParams& p, cudaStream_t s) {
    const int64_t threads = p.rows * GS;
    const int64_t blocks = (threads + kNormThreads - 1) / kNormThreads;
    gdn_gated_rmsnorm_kernel<OT, ZT, GS, kVec><<<(unsigned)blocks, kNormThreads, 0, s>>>(
        static_cast<const OT*>(p.o), static_cast<const ZT*>(p.z), p.w, static_cast<OT*>(p.y), p.rows, p.DV, p.eps, p);
    return cudaGetLastError();
}

template <typename OT, typename ZT, int GS, int NCH>
cudaError_t launch_norm_reg(const GatedNormParams& p, cudaStream_t s) {
    const int64_t threads = p.rows * GS;
    const int64_t blocks = (threads + kNormThreads - 1) / kNormThreads;
    gdn_gated_rmsnorm_reg_kernel<OT, ZT, GS, NCH><<<(unsigned)blocks, kNormThreads, 0, s>>>(
        static_cast<const OT*>(p.o), static_cast<const ZT*>(p.z), p.w, static_cast<OT*>(p.y), p.rows, p.DV, p.eps, p);
    return cudaGetLastError();
}

// 8-column chunks a lane loads at once for rows of up to 32 chunks (more bytes in flight per thread)
#ifndef GDN_NORM_LANE_CHUNKS
#define GDN_NORM_LANE_CHUNKS 1
#endif
constexpr int kLaneChunks = GDN_NORM_LANE_CHUNKS;

template <typename OT, typename ZT>
cudaError_t launch_norm_t(const GatedNormParams& p, cudaStream_t s) {
    if (!p.vec) return launch_norm_gs<OT, ZT, 32, false>(p, s);
    const int chunks = p.DV / 8;  // lanes per row: the chunks of a row over kLaneChunks, a power of two, <= 32
    if (chunks <= kLaneChunks) return launch_norm_reg<OT, ZT, 1, kLaneChunks>(p, s);
    if (chunks <= 2 * kLaneChunks) return launch_norm_reg<OT, ZT, 2, kLaneChunks>(p, s);
    if (chunks <= 4 * kLaneChunks) return launch_norm_reg<OT, ZT, 4, kLaneChunks>(p, s);
    if (chunks <= 8 * kLaneChunks) return launch_norm_reg<OT, ZT, 8, kLaneChunks>(p, s);
    if (chunks <= 16 * kLaneChunks) return launch_norm_reg<OT, ZT, 16, kLaneChunks>(p, s);
    if (chunks <= 32) return launch_norm_reg<OT, ZT, 32, 1>(p, s);
    if (chunks <= 64) return launch_norm_reg<OT, ZT, 32, 2>(p, s);
    if (chunks <= 128) return launch_norm_reg<OT, ZT, 32, 4>(p, s);
    return launch_norm_gs<OT, ZT, 32, true>(p, s);
}

}  // namespace

// The largest row count launch_gated_norm accepts: rows * 32 threads in at most 2^31 - 1 blocks.
int64_t gated_norm_max_rows() { return ((int64_t)0x7fffffff * kNormThreads) / 32; }

cudaError_t launch_gated_norm(const GatedNormParams& p, cudaStream_t s) {
    if (p.o_bf16)
        return p.z_bf16 ? launch_norm_t<__nv_bfloat16, __nv_bfloat16>(p, s) : launch_norm_t<__nv_bfloat16, float>(p, s);
    return p.z_bf16 ? launch_norm_t<float, __nv_bfloat16>(p, s) : launch_norm_t<float, float>(p, s);
}

}  // namespace gdn
