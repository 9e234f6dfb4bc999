// bf16 instantiations of the CUDA-core split-KV attention kernel.
#include "pa_attn_cc.cuh"

namespace pa {
cudaError_t launch_attn_cc_bf16(const AttnParams& p, int head_size, int group, int positions,
                                int num_sms, cudaStream_t stream) {
  return dispatch_cc<__nv_bfloat16>(p, head_size, group, positions, num_sms, stream);
}
}  // namespace pa
