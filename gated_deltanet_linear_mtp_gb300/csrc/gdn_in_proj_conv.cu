// gdn_in_proj_conv.cu -- the in_proj projection of the decode / verify rows with its causal conv1d epilogue, and
// the convolution state's commit (sm_103a).
//
// TensorRT-LLM PR #20937 (GB300 Qwen3.8-Flash-Next NVFP4), What changes, Decode at small batch: "the in_proj GEMV
// with a fused conv1d epilogue, for 2..16 verify rows and up to 8 decode rows"; the convolution state is committed
// with the accepted prefix from the verify rows' recovery records (issue "Proposal: native BF16 MTP speculative
// decoding for dense Qwen3.8-27B", What).  For lane b (rows b*T .. b*T+T-1 of x) and output channel c of W:
//     p[t, c] = sum_h W[c, h] x[b*T + t, h]                         (fp32 accumulation of bf16 products)
//     channels q | k | v (c < Cc): u[t, c] = R_state(p[t, c]); seq = state[slot, 0 .. K-2, c], u[0 .. T-1, c];
//         y[t, c] = bias[c] + sum_j w[c, j] seq[t + j, c], SiLU if asked; decode writes the last K-1 of seq back,
//         verify keeps u as its recovery records
//     channels z | b | a: the projection itself.
//
// gdn_in_proj_conv_kernel: one CTA of 6 warps per (128 output channels, a tile of whole lanes, a slice of the
// hidden dimension).  W is the dense operand: its 128 x 64 boxes and the rows' N x 64 boxes arrive by TMA (128-byte
// swizzle) into a ring of stages (lane 0 of warp 4); lane 0 of warp 5 issues tcgen05.mma (M = 128 channels, N = the
// tile's rows padded to 16, K = 16) into a tensor-memory accumulator of 128 lanes x N columns.  The bytes are W's
// (50 MB for a 12352 x 2048 projection), read once, so a small row count is HBM-bound: the grid splits the hidden
// dimension over a thread-block cluster of up to 8 CTAs, the split chosen from the cluster occupancy on the host,
// and each rank pushes its partial sums into the owning rank's ring (distributed shared memory) once every ring is
// free.  Warps 0-3 are the epilogue (thread = channel, so every load and store of the state, the outputs and the
// records is one coalesced row); they load the taps, indices and state rows they will need while the main loop
// runs, and keep their loops rolled (after an L2 flush the code itself comes from memory).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>

#include "gdn.h"
#include "gdn_internal.h"
#include "gdn_tcgen05.cuh"

namespace gdn {

namespace {

constexpr int kIpM = 128;                  // output channels per tile: the accumulator's tensor-memory lanes
constexpr int kIpKC = 64;                  // hidden columns per stage: one 128-byte swizzled box
constexpr uint32_t kIpWBox = kIpM * kIpKC * 2;  // bytes of W per stage
constexpr int kIpEpiWarps = 4;            // warps 0-3: one per 32 tensor-memory lanes (channels); the epilogue
constexpr int kIpProducerWarp = 4;         // lane 0: the TMA loads
constexpr int kIpMmaWarp = 5;              // lane 0: the MMAs; the warp allocates the tensor memory
constexpr int kIpThreads = 32 * 6;
constexpr int kIpMaxN = 64;                // rows per tile (the MMA's N): more lanes per CTA serialise the epilogue
constexpr int kIpMaxPf = 16;               // lanes whose indices and state rows the epilogue warps gather in advance
constexpr int kIpMaxCluster = 8;
constexpr int kIpMaxStages = 8;
constexpr uint32_t kIpWaitPolls = GDN_WAIT_POLLS;

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void st_cluster(float* local, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared memory, from a 1024-byte aligned base: `stages` x (W box | rows box), then the mbarriers full[stages],
// empty[stages], done, then the tensor-memory address.  The epilogue's partial sums, [ks][lanes a rank owns][T][128]
// fp32, reuse the ring (ring_holds, checked on the host).
__host__ __device__ inline uint32_t ip_stage_bytes(int N) { return kIpWBox + (uint32_t)N * 128u; }
__host__ __device__ inline uint32_t ip_bar_offset(int N, int S) { return ip_stage_bytes(N) * (uint32_t)S; }
__host__ __device__ inline uint32_t ip_tslot_offset(int N, int S) { return ip_bar_offset(N, S) + 8u * (2u * S + 1u); }
// the gathered lane indices [kIpMaxPf] int32, then the gathered state rows [lanes][K - 1][128] (4 bytes a channel)
__host__ __device__ inline uint32_t ip_slots_offset(int N, int S) { return (ip_tslot_offset(N, S) + 4u + 15u) & ~15u; }
__host__ __device__ inline uint32_t ip_pf_offset(int N, int S) { return ip_slots_offset(N, S) + 4u * kIpMaxPf; }
__host__ __device__ inline uint32_t ip_pf_bytes(int lanes, int K) { return (uint32_t)lanes * (K - 1) * kIpM * 4u; }
__host__ __device__ inline uint32_t ip_smem_bytes(int N, int S, int pf_lanes, int K) {
    return ip_pf_offset(N, S) + ip_pf_bytes(pf_lanes, K) + 1024u;  // + alignment slack
}

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ void store_elem(void* base, bool bf16, int64_t i, float v) {
    if (bf16)
        static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
    else
        static_cast<float*>(base)[i] = v;
}

__device__ __forceinline__ float load_elem(const void* base, bool bf16, int64_t i) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]) : static_cast<const float*>(base)[i];
}

}  // namespace

// The launch's tiling: N rows per tile (whole lanes, padded to 16), `ks` ranks splitting the hidden dimension's
// `kchunks` 64-column chunks, `stages` ring stages.
struct IpTiling {
    int N, lanes_per_tile, ks, kchunks, stages;
    int pf_lanes;  // lanes whose indices (and, in tiles of convolved channels, state rows) are gathered in advance
};

// K: convolution taps (2..4)
template <int K>
__global__ void __launch_bounds__(kIpThreads, 1)
    gdn_in_proj_conv_kernel(const InProjConvParams p, const IpTiling g, const __grid_constant__ CUtensorMap wmap,
                            const __grid_constant__ CUtensorMap xmap) {
    extern __shared__ __align__(1024) unsigned char ip_smem[];
    __shared__ int failed;
    const uint32_t raw = smem_u32(ip_smem);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* const gbase = ip_smem + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int rank = blockIdx.x, ctile = blockIdx.y, rtile = blockIdx.z;
    const int N = g.N, S = g.stages;
    const uint32_t stage_b = ip_stage_bytes(N);
    const uint32_t bars = base + ip_bar_offset(N, S);  // full s: + 8 s; empty s: + 8 (S + s); done: + 16 S
    const uint32_t done_bar = bars + 16u * S;
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + ip_tslot_offset(N, S));
    int* const slots_s = reinterpret_cast<int*>(gbase + ip_slots_offset(N, S));
    unsigned char* const pf = gbase + ip_pf_offset(N, S);
    const int c0 = rank * g.kchunks / g.ks, nk = (rank + 1) * g.kchunks / g.ks - c0;  // nk >= 1 (host)
    const uint32_t ncols = N <= 32 ? 32u : N <= 64 ? 64u : N <= 128 ? 128u : 256u;

    const int producer = 32 * kIpProducerWarp;
    if (tid == producer) {
        for (int s = 0; s < 2 * S + 1; ++s) mbar_init(bars + 8u * s, 1);
        fence_mbar_init();
        failed = 0;
    }
    if (warp == kIpMmaWarp) tmem_alloc(smem_u32(tmem_slot), ncols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // The epilogue's inputs do not depend on the product: warps 0-3 (thread = channel c) load the channel's taps and
    // bias and the first owned lane's index and state entries now, so that their latency hides behind the main loop.
    const int64_t c = (int64_t)ctile * kIpM + tid;
    const bool epi = warp < kIpEpiWarps;
    const bool chan = epi && c < p.C, conv = c < p.Cc;
    const int T = p.T;
    const int n_own = rank < g.lanes_per_tile ? (g.lanes_per_tile - rank + g.ks - 1) / g.ks : 0;
    float w[K], bias = 0.f, st0[K - 1];
#pragma unroll
    for (int j = 0; j < K; ++j) w[j] = chan && conv ? p.conv_w[c * K + j] : 0.f;
    if (chan && conv && p.conv_b != nullptr) bias = p.conv_b[c];
    const int b0 = rtile * g.lanes_per_tile + rank;
    const int slot0 = epi && n_own > 0 && b0 < p.B ? p.indices[b0] : -2;  // -2: no lane
#pragma unroll
    for (int j = 0; j < K - 1; ++j)
        st0[j] = chan && conv && slot0 >= 0 && slot0 < p.num_slots
                     ? load_elem(p.state, p.state_bf16, ((int64_t)slot0 * (K - 1) + j) * p.Cc + c)
                     : 0.f;
    // With more lanes per rank (g.pf_lanes > 0): the first pf_n owned lanes' indices into shared memory, then (tiles
    // of convolved channels, 16-byte aligned rows) their state rows by 16-byte cp.async copies, all in flight
    // during the main loop; the epilogue then reads shared memory only.
    const int pf_n = epi ? min(n_own, g.pf_lanes) : 0;
    const bool pf_state = pf_n > 0 && p.state_vec && (int64_t)ctile * kIpM < p.Cc;
    if (pf_n > 0) {
        if (tid < pf_n) {
            const int b = b0 + tid * g.ks;
            slots_s[tid] = b < p.B ? p.indices[b] : -2;
        }
        named_sync(1, 32 * kIpEpiWarps);
        if (pf_state) {
            const int eb = p.state_bf16 ? 2 : 4;
            const int cpr = (int)min((int64_t)kIpM, p.Cc - (int64_t)ctile * kIpM) * eb / 16;  // chunks of a row
            const unsigned char* const src0 =
                static_cast<const unsigned char*>(p.state) + (int64_t)ctile * kIpM * eb;
            for (int i = tid; i < pf_n * (K - 1) * cpr; i += 32 * kIpEpiWarps) {
                const int m = i / ((K - 1) * cpr), r = i - m * ((K - 1) * cpr), j = r / cpr, q = r - j * cpr;
                const int sl = slots_s[m];
                if (sl >= 0 && sl < p.num_slots)
                    cp_async16(smem_u32(pf + ((m * (K - 1) + j) * kIpM) * eb + q * 16),
                               src0 + (((int64_t)sl * (K - 1) + j) * p.Cc) * eb + q * 16);
            }
            cp_async_commit();
        }
    }

    // roles by whole warps: lane 0 of the producer warp loads, lane 0 of the MMA warp issues the MMAs, the other
    // lanes of those warps wait at __syncwarp (a lane polling beside them would take their issue slots)
    int issued = 0;  // producer: loads issued
    if (tid == producer) {
        // one stage = W's 128 x 64 box and the tile's N x 64 rows box, on the stage's full barrier
        const int row0 = rtile * g.lanes_per_tile * p.T;
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            if (i >= S && !mbar_wait_bounded(bars + 8u * (S + s), (uint32_t)((i / S) - 1) & 1u, kIpWaitPolls)) {
                failed = 1;
                break;
            }
            const uint32_t dst = base + (uint32_t)s * stage_b;
#ifdef GDN_TEST_MISSING_COPY
            // test build: the first stage of CTA (0, 0, 0) is never loaded (nor arrived on), so the waits for it
            // and for its reuse run out
            if (i == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) continue;
#endif
            mbar_arrive_expect_tx(bars + 8u * s, stage_b);
            tma_load_2d(dst, &wmap, (c0 + i) * kIpKC, ctile * kIpM, bars + 8u * s);
            tma_load_2d(dst + kIpWBox, &xmap, (c0 + i) * kIpKC, row0, bars + 8u * s);
            issued = i + 1;
        }
    } else if (tid == 32 * kIpMmaWarp) {
        // D[128 x N] (+)= W box . rows box^T, four K = 16 steps per stage; each stage's completion frees it for the
        // producer, the last one signals the epilogue
        const uint32_t idesc = umma_idesc_bf16(kIpM, N);
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            if (!mbar_wait_bounded(bars + 8u * s, (uint32_t)(i / S) & 1u, kIpWaitPolls)) {
                failed = 1;
                break;
            }
            tc_fence_after();
            const uint32_t a = base + (uint32_t)s * stage_b, b = a + kIpWBox;
#pragma unroll
            for (int kk = 0; kk < kIpKC / 16; ++kk)
                umma_bf16(tmem, umma_desc_sw128(a + 32u * kk), umma_desc_sw128(b + 32u * kk), idesc,
                          (i | kk) != 0 ? 1u : 0u);
            umma_commit(bars + 8u * (S + s));
        }
        umma_commit(done_bar);
    }
    if (!epi) __syncwarp();
    if (epi && !mbar_wait_bounded(done_bar, 0, kIpWaitPolls)) failed = 1;
    tc_fence_after();
    __syncthreads();
    const bool ok = failed == 0;
    if (!ok) {
        // a wait ran out: let the MMAs and the copies already issued finish before the memory is reused or freed
        if (tid == producer) {
            mbar_wait_bounded(done_bar, 0, kIpWaitPolls);
            for (int i = issued > S ? issued - S : 0; i < issued; ++i)
                mbar_wait_bounded(bars + 8u * (i % S), (uint32_t)(i / S) & 1u, kIpWaitPolls);
            if (p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_TIMEOUT);
        }
        __syncthreads();
    }

    // The partial sums to their owners.  Lane li of the tile belongs to rank li mod ks (as its m = li / ks-th lane);
    // every rank writes its accumulator column (li, t) into the owner's ring as part[src = rank][m][t][channel]
    // (thread = channel = tensor-memory lane 32 warp + lane): remote stores for the other ranks, which cost no round
    // trip.  A first cluster barrier makes sure every rank's main loop is done with its ring, a second that every
    // partial has arrived; after it all reads are local.
    const int mmax = (g.lanes_per_tile + g.ks - 1) / g.ks;  // lanes a rank owns at most
    float* const part = reinterpret_cast<float*>(gbase);     // [ks][mmax][T][128]
    if (g.ks > 1) cluster_barrier();
    if (ok && epi) {
        int li = 0, t = 0, owner = 0, m = 0;  // lane, row, owning rank and its lane index of column col + j
        for (int col = 0; col < N; col += 16) {
            float f[16];
            tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)col, f);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (li < g.lanes_per_tile) {
                    float* const e = part + (((rank * mmax + m) * T + t) * kIpM + tid);
                    if (owner == rank)
                        *e = f[j];
                    else
                        st_cluster(e, (uint32_t)owner, f[j]);
                }
                if (++t == T) {
                    t = 0;
                    ++li;
                    if (++owner == g.ks) {
                        owner = 0;
                        ++m;
                    }
                }
            }
        }
    }
    if (pf_state) cp_async_wait_all();  // the gathered state rows, before the barrier publishes them
    tc_fence_before();
    __syncthreads();
    if (g.ks > 1) cluster_barrier();  // every partial is in its owner's ring

    // each rank takes lanes rank, rank + ks, ... of the tile (the first one's loads went out before the main loop);
    // thread = channel c.  The loops are kept rolled: after an L2 flush the code is fetched from memory too.
    // where the channel's values go: q | k (HK * DK each), v (HV * DV); z (HV * DV), b, a (HV each)
    const int64_t qc = (int64_t)p.HK * p.DK, vc = (int64_t)p.HV * p.DV, cz = c - p.Cc;
    void* dst;
    int64_t dc, dstride;
    if (conv) {
        dst = c < qc ? p.q : c < 2 * qc ? p.k : p.v;
        dc = c < qc ? c : c < 2 * qc ? c - qc : c - 2 * qc;
        dstride = c < 2 * qc ? qc : vc;
    } else {
        dst = cz < vc ? p.z : cz < vc + p.HV ? p.bo : p.ao;
        dc = cz < vc ? cz : cz < vc + p.HV ? cz - vc : cz - vc - p.HV;
        dstride = cz < vc ? vc : p.HV;
    }
#pragma unroll 1
    for (int m = 0; ok && epi && m < n_own; ++m) {
        const int b = b0 + m * g.ks;
        int slot = slot0;
        float st[K - 1];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) st[j] = st0[j];
        if (m < pf_n) {
            slot = slots_s[m];
#pragma unroll
            for (int j = 0; j < K - 1; ++j)
                st[j] = pf_state && chan && conv && slot >= 0 && slot < p.num_slots
                            ? (p.state_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(pf)[(m * (K - 1) + j) * kIpM + tid])
                                            : reinterpret_cast<const float*>(pf)[(m * (K - 1) + j) * kIpM + tid])
                            : st[j];
            if (!pf_state && m > 0) {
#pragma unroll
                for (int j = 0; j < K - 1; ++j)
                    st[j] = chan && conv && slot >= 0 && slot < p.num_slots
                                ? load_elem(p.state, p.state_bf16, ((int64_t)slot * (K - 1) + j) * p.Cc + c)
                                : 0.f;
            }
        } else if (m > 0) {
            slot = b < p.B ? p.indices[b] : -2;
#pragma unroll
            for (int j = 0; j < K - 1; ++j)
                st[j] = chan && conv && slot >= 0 && slot < p.num_slots
                            ? load_elem(p.state, p.state_bf16, ((int64_t)slot * (K - 1) + j) * p.Cc + c)
                            : 0.f;
        }
        if (slot < 0 || slot >= p.num_slots) {
            if (slot != -1 && slot != -2 && ctile == 0 && tid == 0 && p.err != nullptr) atomicOr(p.err, GDN_ERRBIT_INDEX);
            continue;
        }
        if (!chan) continue;
        // the full sums over the ranks (in rank order), rounded to the state type for the convolved channels, into
        // the src = 0 slot: only this thread reads them from here on
        float* const u = part + (m * T) * kIpM + tid;  // u[t * kIpM]
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
            float v = u[t * kIpM];
            for (int r = 1; r < g.ks; ++r) v += part[((r * mmax + m) * T + t) * kIpM + tid];
            if (conv && p.state_bf16) v = round_bf16(v);
            u[t * kIpM] = v;
        }
        const int64_t row0 = (int64_t)b * T;
        if (!conv) {
#pragma unroll 1
            for (int t = 0; t < T; ++t) store_elem(dst, p.out_bf16, (row0 + t) * dstride + dc, u[t * kIpM]);
            continue;
        }
        // the convolution over seq = state (K - 1 entries, oldest first), u[0 .. T-1]
        auto seq = [&](int i) -> float {
            if (i >= K - 1) return u[(i - (K - 1)) * kIpM];
            float x = st[0];
#pragma unroll
            for (int j = 1; j < K - 1; ++j)
                if (i == j) x = st[j];
            return x;
        };
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
            float y = bias;
#pragma unroll
            for (int j = 0; j < K; ++j) y = fmaf(w[j], seq(t + j), y);
            if (p.silu) y = y / (1.f + expf(-y));
            store_elem(dst, p.out_bf16, (row0 + t) * dstride + dc, y);
            if (p.records != nullptr) store_elem(p.records, p.state_bf16, (row0 + t) * p.Cc + c, u[t * kIpM]);
        }
        if (p.write_state) {
            float nw[K - 1];
#pragma unroll
            for (int j = 0; j < K - 1; ++j) nw[j] = seq(T + j);  // every read before the first write
#pragma unroll
            for (int j = 0; j < K - 1; ++j)
                store_elem(p.state, p.state_bf16, ((int64_t)slot * (K - 1) + j) * p.Cc + c, nw[j]);
        }
    }

    // (no final cluster barrier: every remote store came before the one above, so no rank touches another's
    // shared memory from there on and each may leave when it is done)
    __syncthreads();
    if (warp == kIpMmaWarp) tmem_dealloc(tmem, ncols);
}

// The convolution state after each lane's first L accepted rows: pool[slot, j, c] = seq[L + j, c] with seq = the
// slot's K - 1 entries, then the lane's T recovery records (bit copies: both are stored values of the state type).
// One thread per (lane, channel); every read comes before the first write.
template <typename StT>
__global__ void __launch_bounds__(256) gdn_conv_commit_kernel(const ConvCommitParams p) {
    const int b = blockIdx.y;
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool reporter = threadIdx.x == 0 && blockIdx.x == 0 && p.err != nullptr;
    const int slot = p.indices[b];
    if (slot < 0 || slot >= p.num_slots) {
        if (slot != -1 && reporter) atomicOr(p.err, GDN_ERRBIT_INDEX);
        return;
    }
    const int L = p.accept_len[b];
    if (L < 0 || L > p.T) {
        if (reporter) atomicOr(p.err, GDN_ERRBIT_ACCEPT_LEN);
        return;
    }
    if (L == 0 || c >= p.Cc) return;
    const int K1 = p.K - 1;  // 1 .. 3
    StT* const st = static_cast<StT*>(p.state) + (int64_t)slot * K1 * p.Cc + c;
    const StT* const rec = static_cast<const StT*>(p.records) + (int64_t)b * p.T * p.Cc + c;
    StT nv[3];
#pragma unroll
    for (int j = 0; j < 3; ++j)
        if (j < K1) nv[j] = L + j < K1 ? st[(int64_t)(L + j) * p.Cc] : rec[(int64_t)(L + j - K1) * p.Cc];
#pragma unroll
    for (int j = 0; j < 3; ++j)
        if (j < K1) st[(int64_t)j * p.Cc] = nv[j];
}

namespace {

bool encode_rows_map(CUtensorMap* map, const void* ptr, int cols, int64_t rows, int box_rows) {
    const EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kIpKC, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Tiling.  A tile holds whole lanes: all B of them when B * T <= 256 rows, else 256 / T.  The ring takes 2..8
// stages within what three CTAs per SM leave (N <= 32), two (N <= 64), or one.  The hidden dimension is split
// over ks ranks (a cluster), ks chosen to minimise waves x chunks per CTA, where a wave is the clusters the GPU
// holds at once (the occupancy calculator: a cluster's CTAs must share a GPC, so 2 x 152 CTA slots do not take
// 2 x 152 / ks clusters); ties go to the smaller ks (less reduction).
// the ring holds the epilogue's partial sums of a split into g.ks ranks
bool ring_holds(const IpTiling& g, int T) {
    const uint64_t mmax = (uint64_t)(g.lanes_per_tile + g.ks - 1) / g.ks;
    return (uint64_t)g.stages * ip_stage_bytes(g.N) >= (uint64_t)g.ks * mmax * T * kIpM * 4;
}

// everything but the split, from the shape alone
// Row tiles: all lanes in one up to 32 rows; two tiles up to 128 rows (64 rows in one tile measured 40 us against
// 27 us in two of 32; more tiles re-read W from L2: 128 rows in four tiles 60 us against 52 us in two); 64-row
// tiles beyond.  N <= 32: three CTAs per SM, the first owned lane prefetched in registers; N = 48 or 64: two, up
// to kIpMaxPf lanes gathered in shared memory.
IpTiling base_tiling(int B, int T, int H, int K) {
    IpTiling g{};
    const int64_t rows = (int64_t)B * T;
    g.lanes_per_tile = rows <= 32 ? B : rows <= 2 * kIpMaxN ? std::min((B + 1) / 2, kIpMaxN / T) : kIpMaxN / T;
    g.N = (g.lanes_per_tile * T + 15) / 16 * 16;
    g.kchunks = (H + kIpKC - 1) / kIpKC;
    g.pf_lanes = g.N <= 32 ? 0 : std::min(g.lanes_per_tile, kIpMaxPf);
    const uint32_t budget = (g.N <= 32 ? 72u * 1024u : 110u * 1024u) - ip_pf_bytes(g.pf_lanes, K);
    g.stages = (int)std::min<uint32_t>(kIpMaxStages, std::max<uint32_t>(2, budget / ip_stage_bytes(g.N)));
    g.ks = 1;
    return g;
}

template <int K>
IpTiling in_proj_tiling(int B, int T, int H, int64_t C) {
    IpTiling g = base_tiling(B, T, H, K);
    const int64_t tiles = ((C + kIpM - 1) / kIpM) * (int64_t)((B + g.lanes_per_tile - 1) / g.lanes_per_tile);
    const uint32_t smem = ip_smem_bytes(g.N, g.stages, g.pf_lanes, K);
    int64_t best = INT64_MAX;
    for (int ks = 1; ks <= std::min(kIpMaxCluster, g.kchunks); ++ks) {
        IpTiling c = g;
        c.ks = ks;
        if (!ring_holds(c, T)) continue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ks, (unsigned)((C + kIpM - 1) / kIpM), 1);
        cfg.blockDim = dim3(kIpThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)ks;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, gdn_in_proj_conv_kernel<K>, &cfg) != cudaSuccess ||
            clusters < 1) {
            (void)cudaGetLastError();
            continue;
        }
        const int64_t cost = ((tiles + clusters - 1) / clusters) * ((g.kchunks + ks - 1) / ks);
        if (cost < best) {
            best = cost;
            g.ks = ks;
        }
    }
    return g;
}

// The split last chosen on each device (one cache per K), with a hash of its (B, T, H, C) in the same word: the occupancy
// queries run once per shape.  Only ks is cached, clamped to the shape's chunks on the way out, so a stale or
// colliding entry can cost speed but never correctness.
template <int K>
IpTiling cached_tiling(int B, int T, int H, int64_t C) {
    static std::atomic<uint64_t> cache[64];  // hash << 8 | ks; zero (static): empty
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return in_proj_tiling<K>(B, T, H, C);
    const uint64_t h = (((uint64_t)B * 0x9E3779B97F4A7C15ull) ^ ((uint64_t)T << 40) ^ ((uint64_t)H << 20) ^
                        (uint64_t)C) & 0x00FFFFFFFFFFFFFFull;
    const uint64_t c = cache[dev].load(std::memory_order_relaxed);
    if (c != 0 && (c >> 8) == h) {
        IpTiling g = base_tiling(B, T, H, K);
        g.ks = std::max(1, std::min<int>((int)(c & 0xffu), std::min(kIpMaxCluster, g.kchunks)));
        while (g.ks > 1 && !ring_holds(g, T)) --g.ks;
        return g;
    }
    const IpTiling g = in_proj_tiling<K>(B, T, H, C);
    cache[dev].store(h << 8 | (uint64_t)g.ks, std::memory_order_relaxed);
    return g;
}

template <int K>
cudaError_t launch_in_proj_k(const InProjConvParams& p, const CUtensorMap& wmap, cudaStream_t s) {
    auto kernel = gdn_in_proj_conv_kernel<K>;
    // the ring of this shape (the split does not change it), opened before the occupancy queries see the kernel
    const IpTiling b = base_tiling(p.B, p.T, p.H, K);
    const uint32_t smem = ip_smem_bytes(b.N, b.stages, b.pf_lanes, K);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const IpTiling g = cached_tiling<K>(p.B, p.T, p.H, p.C);
    if (!ring_holds(g, p.T)) return cudaErrorInvalidConfiguration;  // ks = 1 always fits: lanes x T <= N
    CUtensorMap xmap;
    if (!encode_rows_map(&xmap, p.x, p.H, (int64_t)p.B * p.T, g.N)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)g.ks, (unsigned)((p.C + kIpM - 1) / kIpM),
                       (unsigned)((p.B + g.lanes_per_tile - 1) / g.lanes_per_tile));
    cfg.blockDim = dim3(kIpThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)g.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p, g, wmap, xmap);
}

cudaError_t launch_in_proj_conv(const InProjConvParams& p, cudaStream_t s) {
    if (p.B == 0) return cudaSuccess;
    CUtensorMap wmap;
    if (!encode_rows_map(&wmap, p.W, p.H, p.C, kIpM)) return cudaErrorInvalidValue;
    switch (p.K) {
    case 2: return launch_in_proj_k<2>(p, wmap, s);
    case 3: return launch_in_proj_k<3>(p, wmap, s);
    case 4: return launch_in_proj_k<4>(p, wmap, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_conv_commit(const ConvCommitParams& p, cudaStream_t s) {
    if (p.B == 0) return cudaSuccess;
    const dim3 grid((unsigned)((p.Cc + 255) / 256), (unsigned)p.B);
    if (p.state_bf16)
        gdn_conv_commit_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p);
    else
        gdn_conv_commit_kernel<float><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
