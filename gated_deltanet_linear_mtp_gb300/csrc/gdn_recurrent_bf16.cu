// Instances of the decode / verify kernel for a bf16 state pool (q/k/v in fp32 or bf16).
#include "gdn_recurrent_launch.cuh"

namespace gdn {

cudaError_t launch_recurrent_bf16state(const RecurrentParams& p, int B, int DK, bool qkv_bf16, cudaStream_t s) {
    return qkv_bf16 ? launch_recurrent<__nv_bfloat16, __nv_bfloat16>(p, B, DK, s)
                    : launch_recurrent<float, __nv_bfloat16>(p, B, DK, s);
}

bool chunked_verify_eligible(int B, int T, int DK, int DV, int HV, int num_slots) {
    return chunked_range(B, T, DK, DV, HV, num_slots);
}

bool launch_replay_verify_bf16state(const RecurrentParams& p, int B, int DK, bool qkv_bf16, cudaStream_t s,
                                    cudaError_t& err) {
    return qkv_bf16 ? launch_replay_verify<__nv_bfloat16>(p, B, DK, s, err) : launch_replay_verify<float>(p, B, DK, s, err);
}

}  // namespace gdn
