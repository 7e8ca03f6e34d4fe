// gdn_recurrent_launch.cuh -- launches the decode / verify kernel for one (q/k/v type, state type) pair:
// grid = (ceil(DV / RPC), HV, B), one CTA of Split<DK>::THREADS per (lane, value head, block of RPC rows).
#pragma once

#include "gdn_recurrent.cuh"

namespace gdn {

template <typename InT, typename StT, int DK>
cudaError_t launch_dk(const RecurrentParams& p, int B, cudaStream_t s) {
    constexpr int RPC = Split<DK>::RPC;
    const size_t smem = sizeof(float) * general_smem_floats(DK, RPC, p.T);
    const dim3 grid((p.DV + RPC - 1) / RPC, p.HV, B);
    gdn_recurrent_kernel<DK, InT, StT><<<grid, Split<DK>::THREADS, smem, s>>>(p);
    return cudaGetLastError();
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
