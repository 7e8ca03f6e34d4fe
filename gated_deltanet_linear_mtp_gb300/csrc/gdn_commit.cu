// gdn_commit.cu -- accepted-prefix commit: pool[idx[b], :] = cache[b, L_b - 1, :] (all heads of one lane
// are one contiguous run of HV * DV * DK elements on both sides), a bit-exact copy.
//
// HBM-bound copy: each CTA moves kCommitUnroll * 256 * 16 bytes of one lane; every thread issues all of its
// 16-byte loads before its stores so that each SM keeps many bytes in flight.  Loads take the read-only
// path without L1 allocation; stores are plain (the pool is read again by the next step).
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {

constexpr int kCommitThreads = 256;
constexpr int kCommitUnroll = 4;
constexpr int64_t kCommitBytesPerCta = (int64_t)kCommitThreads * kCommitUnroll * 16;

__device__ __forceinline__ uint4 ld_ro16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__global__ void __launch_bounds__(kCommitThreads) gdn_commit_kernel(const CommitParams p) {
    const int b = blockIdx.y;
    const int slot = p.indices[b];
    const bool first = threadIdx.x == 0 && blockIdx.x == 0;
    if (slot < 0 || slot >= p.num_slots) {
        if (slot != -1 && first && p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_INDEX);
        return;
    }
    const int L = p.accept_len[b];
    if (L < 0 || L > p.T) {
        if (first && p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_ACCEPT_LEN);
        return;
    }
    if (L == 0) return;
    const char* src = static_cast<const char*>(p.cache) + ((int64_t)b * p.T + (L - 1)) * p.lane_bytes;
    char* dst = static_cast<char*>(p.pool) + (int64_t)slot * p.lane_bytes;
    const int64_t base = (int64_t)blockIdx.x * kCommitBytesPerCta + (int64_t)threadIdx.x * 16;
    uint4 r[kCommitUnroll];
#pragma unroll
    for (int u = 0; u < kCommitUnroll; ++u) {
        const int64_t off = base + (int64_t)u * kCommitThreads * 16;
        if (off < p.lane_bytes) r[u] = ld_ro16(src + off);
    }
#pragma unroll
    for (int u = 0; u < kCommitUnroll; ++u) {
        const int64_t off = base + (int64_t)u * kCommitThreads * 16;
        if (off < p.lane_bytes)
            asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(dst + off), "r"(r[u].x), "r"(r[u].y),
                         "r"(r[u].z), "r"(r[u].w)
                         : "memory");
    }
}

cudaError_t launch_commit(const CommitParams& p, int B, cudaStream_t s) {
    const int64_t blocks = (p.lane_bytes + kCommitBytesPerCta - 1) / kCommitBytesPerCta;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    gdn_commit_kernel<<<dim3((unsigned)blocks, B), kCommitThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
