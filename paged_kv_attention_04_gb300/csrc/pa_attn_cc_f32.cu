// fp32 instantiations of the CUDA-core split-KV attention kernel.
#include "pa_attn_cc.cuh"

namespace pa {
cudaError_t launch_attn_cc_f32(const AttnParams& p, int head_size, int group, int positions,
                               int num_sms, cudaStream_t stream, int* grid_only) {
  return dispatch_cc<float>(p, head_size, group, positions, num_sms, stream, grid_only);
}
}  // namespace pa
