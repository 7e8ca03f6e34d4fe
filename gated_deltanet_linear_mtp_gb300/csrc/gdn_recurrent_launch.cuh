// gdn_recurrent_launch.cuh -- picks and launches the decode / verify / replay-commit kernel for one
// (q/k/v type, state type) pair.
//
//   gdn_recurrent_staged_kernel, grid = (ceil(DV / (NSUB * RPC)), HV, B), when a CTA has little work per
//       state byte (T * sizeof(state) <= 8: bf16 with T <= 4, fp32 with T <= 2), so that the state's load
//       latency dominates and bulk copies keep more bytes in flight, and when that grid still gives every
//       SM at least two CTAs.  A CTA stages 16 KiB of state for an fp32 pool or T >= 4, 32 KiB otherwise
//       (and the fp32 16 KiB kernel at DK = 128 budgets registers for 7 CTAs per SM instead of 6);
//   gdn_recurrent_kernel, grid = (ceil(DV / RPC), HV, B), otherwise.
// The rules follow B x T x state-dtype sweeps on the GB300: the staged kernel was 15-40% faster than the
// direct one inside its rule and 4-80% slower outside it; 16 KiB stages were up to 15% faster than 32 KiB
// for fp32 pools and bf16 with T = 4, and up to 12% slower for bf16 with T <= 2.  Both kernels run
// Split<DK>::THREADS threads per CTA.
// On a bf16 pool with T <= 8 and DK >= 64, a verify that stores neither intermediate states nor a write-back,
// and a replay commit, run the persistent chunked tensor-core kernel (gdn_verify_chunked.cuh) instead, one CTA
// per resident slot of the GPU.
#pragma once

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <type_traits>

#include "gdn_recurrent.cuh"
#include "gdn_verify_chunked.cuh"

namespace gdn {

// The chunked kernel takes T <= 8 tokens and DK >= 64; it addresses num_slots * HV heads with a signed 32-bit
// TMA coordinate and counts its items in int.  Beyond these, the token-by-token kernels serve the call.
inline bool chunked_range(int B, int T, int DK, int DV, int HV, int num_slots) {
    const uint64_t heads = (uint64_t)num_slots * (uint64_t)HV;
    const uint64_t items = (uint64_t)B * HV * (((uint64_t)DV + kChunkRows - 1) / kChunkRows);
    return T >= 1 && T <= kChunkMaxT && DK >= kChunkMinDK && heads <= INT32_MAX && items <= INT32_MAX;
}

constexpr int kStagedMaxTokenBytes = 8;  // T * sizeof(state element) at or below which staging pays
constexpr int kStagedMinCtasPerSm = 2;

inline int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

template <typename StT, int DK, int KIB>
bool use_staged(const RecurrentParams& p, int B, int sms) {
    using ST = Staged<DK, StT, KIB>;
    if (sms <= 0 || p.T * (int)sizeof(StT) > kStagedMaxTokenBytes) return false;
    const int64_t ctas = (int64_t)B * p.HV * ((p.DV + ST::ROWS - 1) / ST::ROWS);
    return ctas >= (int64_t)kStagedMinCtasPerSm * sms;
}

// A kernel whose CTAs of one (lane, head) run as a thread-block cluster of grid.x (the fused gated norm).
template <typename Kernel>
cudaError_t launch_head_cluster(Kernel kernel, dim3 grid, int threads, size_t smem, cudaStream_t s,
                                const RecurrentParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = grid.x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// The standalone gated norm of the outputs the kernel just stored (rows of padded or invalid lanes untouched):
// the fused norm's fallback where a head spans more CTAs than one cluster takes, or the grid more than one wave.
inline cudaError_t launch_norm_after(const RecurrentParams& p, int B, cudaStream_t s) {
    auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    GatedNormParams g{};
    g.o = p.o;
    g.z = p.nz;
    g.w = p.nw;
    g.y = p.ny;
    g.rows = (int64_t)B * p.T * p.HV;
    g.DV = p.DV;
    g.o_bf16 = p.out_bf16;
    g.z_bf16 = p.nz_bf16;
    g.vec = p.DV % 8 == 0 && a16(p.o) && a16(p.nz) && a16(p.ny) && a16(p.nw);
    g.eps = p.neps;
    g.lane_slot = p.indices;
    g.rows_per_lane = (int64_t)p.T * p.HV;
    g.num_slots = p.num_slots;
    return launch_gated_norm(g, s);
}

// CTAs of `kernel` (threads, smem bytes each) resident on one SM of the current device, from the occupancy
// calculator; one cached answer per kernel instance and device (its last smem size), 0 if a query failed
template <typename Kernel>
int resident_ctas_per_sm(Kernel kernel, int threads, size_t smem) {
    static std::atomic<uint64_t> cache[kChunkCachedDevices];  // (smem + 1) << 8 | CTAs; zero (static): none
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cached = dev >= 0 && dev < kChunkCachedDevices;
    if (cached) {
        const uint64_t c = cache[dev].load(std::memory_order_relaxed);
        if ((c >> 8) == (uint64_t)smem + 1) return (int)(c & 0xffu);
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    n = std::min(n, 255);
    if (cached) cache[dev].store(((uint64_t)smem + 1) << 8 | (uint64_t)n, std::memory_order_relaxed);
    return n;
}

// A kernel of the rank-1 family with grid `grid`: with the norm fused (p.nz set), or plain and then the standalone
// norm (p.nz set), or plain.  The norm is fused while a head's CTAs fit one cluster and the whole grid is resident
// at once (one wave).  Past one wave the two launches measured faster on the GB300 (B x pool-dtype sweeps of
// decode and T = 4 verify): each CTA keeps its SM slot through the epilogue, waiting on the slowest CTA of its
// cluster, while the next CTA's state load could use it; inside one wave the fused launch saved 2-3 us of the
// norm's own launch.
template <typename KPlain, typename KNorm>
cudaError_t launch_rank1(KPlain plain, KNorm fused, dim3 grid, int threads, size_t smem, size_t smem_norm,
                         const RecurrentParams& p, int B, cudaStream_t s) {
    if (p.nz != nullptr && grid.x <= (unsigned)kNormMaxCluster) {
        if (smem_norm > 48 * 1024) {
            const cudaError_t e = cudaFuncSetAttribute(fused, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_norm);
            if (e != cudaSuccess) return e;
        }
        const int64_t ctas = (int64_t)grid.x * grid.y * grid.z;
        if (ctas <= (int64_t)sm_count() * resident_ctas_per_sm(fused, threads, smem_norm))
            return launch_head_cluster(fused, grid, threads, smem_norm, s, p);
    }
    RecurrentParams q = p;
    q.nz = nullptr;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(plain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    plain<<<grid, threads, smem, s>>>(q);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && p.nz != nullptr) e = launch_norm_after(p, B, s);
    return e;
}

// the staged kernel with KIB KiB per CTA, if the rule above picks it; false: use the direct kernel
template <typename InT, typename StT, int DK, int KIB>
bool launch_staged(const RecurrentParams& p, int B, int sms, cudaStream_t s, cudaError_t& err) {
    if (!use_staged<StT, DK, KIB>(p, B, sms)) return false;
    using ST = Staged<DK, StT, KIB>;
    const dim3 grid((p.DV + ST::ROWS - 1) / ST::ROWS, p.HV, B);
    err = launch_rank1(gdn_recurrent_staged_kernel<DK, InT, StT, KIB, false>,
                       gdn_recurrent_staged_kernel<DK, InT, StT, KIB, true>, grid, Split<DK>::THREADS,
                       ST::smem_bytes(p.T), NormSmem::end(ST::norm_offset(p.T), p.T, ST::ROWS), p, B, s);
    return true;
}

template <typename InT, typename StT, int DK>
cudaError_t launch_dk(const RecurrentParams& p, int B, cudaStream_t s) {
    constexpr int NT = Split<DK>::THREADS;
    if constexpr (std::is_same<StT, __nv_bfloat16>::value && DK >= kChunkMinDK) {
        const bool verify_only = p.cache == nullptr && p.pool_out == nullptr && p.steps == nullptr;
        const bool replay_commit = p.cache == nullptr && p.pool_out != nullptr && p.steps != nullptr && p.o == nullptr;
        if ((verify_only || replay_commit) && chunked_range(B, p.T, DK, p.DV, p.HV, p.num_slots))
            return replay_commit ? launch_chunked<DK, InT, kModeReplay>(p, B, s)
                                 : launch_chunked<DK, InT, kModeVerify>(p, B, s);
    }
    const int sms = sm_count();
    cudaError_t err = cudaSuccess;
    bool staged;
    if constexpr (std::is_same<StT, float>::value)
        staged = launch_staged<InT, StT, DK, 16>(p, B, sms, s, err);
    else
        staged = p.T >= 4 ? launch_staged<InT, StT, DK, 16>(p, B, sms, s, err)
                          : launch_staged<InT, StT, DK, 32>(p, B, sms, s, err);
    if (staged) return err;
    constexpr int RPC = Split<DK>::RPC;
    const size_t smem = direct_smem_bytes<DK>(p.T);
    const dim3 grid((p.DV + RPC - 1) / RPC, p.HV, B);
    return launch_rank1(gdn_recurrent_kernel<DK, InT, StT, false>, gdn_recurrent_kernel<DK, InT, StT, true>, grid, NT,
                        smem, NormSmem::end(smem, p.T, RPC), p, B, s);
}

// the chunked kernel's replay commit + verify mode, if the call is in its range
template <typename InT, int DK>
bool launch_replay_verify_dk(const RecurrentParams& p, int B, cudaStream_t s, cudaError_t& err) {
    if constexpr (DK >= kChunkMinDK) {
        if (chunked_range(B, p.T, DK, p.DV, p.HV, p.num_slots) && p.T <= kFusedMaxT && p.rT >= 1 &&
            p.rT <= kFusedMaxT) {
            err = launch_chunked<DK, InT, kModeReplayVerify>(p, B, s);
            return true;
        }
    }
    return false;
}

template <typename InT>
bool launch_replay_verify(const RecurrentParams& p, int B, int DK, cudaStream_t s, cudaError_t& err) {
    switch (DK) {
    case 64: return launch_replay_verify_dk<InT, 64>(p, B, s, err);
    case 128: return launch_replay_verify_dk<InT, 128>(p, B, s, err);
    case 256: return launch_replay_verify_dk<InT, 256>(p, B, s, err);
    default: return false;
    }
}

template <typename InT, typename StT>
cudaError_t launch_recurrent(const RecurrentParams& p, int B, int DK, cudaStream_t s) {
    switch (DK) {
    case 16: return launch_dk<InT, StT, 16>(p, B, s);
    case 32: return launch_dk<InT, StT, 32>(p, B, s);
    case 64: return launch_dk<InT, StT, 64>(p, B, s);
    case 128: return launch_dk<InT, StT, 128>(p, B, s);
    case 256: return launch_dk<InT, StT, 256>(p, B, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
