// Attention over an FP8 (E4M3) KV cache with bf16 q/out: the tensor-core
// split-KV kernel with its FP8 staging (codes widened to f16 in shared
// memory; the K scale is folded into the softmax scale, the V scale into the
// final normalisation).
#include "pa_attn_mma.cuh"

#ifndef PA_MMA_FP8_WARPS
#define PA_MMA_FP8_WARPS 4
#endif
#ifndef PA_MMA_FP8_STAGES
#define PA_MMA_FP8_STAGES 2
#endif

namespace pa {

namespace {
template <int D, int G>
cudaError_t dispatch_positions_fp8(const AttnParams& p, int positions, int num_sms,
                                   cudaStream_t stream, int* grid_only) {
  // decode tiles with the keys as M (three CTAs per SM): measured faster than
  // query rows as M for every FP8 workload
  if (positions == 1)
    return launch_mma<D, G, 1, PA_MMA_FP8_WARPS, PA_MMA_FP8_STAGES, true, true>(p, num_sms,
                                                                                stream, grid_only);
  return launch_mma<D, G, kSmallRows / G, PA_MMA_FP8_WARPS, PA_MMA_FP8_STAGES, true>(
      p, num_sms, stream, grid_only);
}

template <int D>
cudaError_t dispatch_group_fp8(const AttnParams& p, int group, int positions, int num_sms,
                               cudaStream_t stream, int* grid_only) {
  switch (group) {
    case 1: return dispatch_positions_fp8<D, 1>(p, positions, num_sms, stream, grid_only);
    case 2: return dispatch_positions_fp8<D, 2>(p, positions, num_sms, stream, grid_only);
    case 4: return dispatch_positions_fp8<D, 4>(p, positions, num_sms, stream, grid_only);
    case 8: return dispatch_positions_fp8<D, 8>(p, positions, num_sms, stream, grid_only);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_attn_fp8(const AttnParams& p, int head_size, int group, int positions,
                            int num_sms, cudaStream_t stream, int* grid_only) {
  switch (head_size) {
    case 64: return dispatch_group_fp8<64>(p, group, positions, num_sms, stream, grid_only);
    case 128: return dispatch_group_fp8<128>(p, group, positions, num_sms, stream, grid_only);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
