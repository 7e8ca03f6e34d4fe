// Instances of the decode / verify kernel for an fp32 state pool (q/k/v in fp32 or bf16).
#include "gdn_recurrent_launch.cuh"

namespace gdn {

cudaError_t launch_recurrent_f32state(const RecurrentParams& p, int B, int DK, bool qkv_bf16, cudaStream_t s) {
    return qkv_bf16 ? launch_recurrent<__nv_bfloat16, float>(p, B, DK, s) : launch_recurrent<float, float>(p, B, DK, s);
}

}  // namespace gdn
