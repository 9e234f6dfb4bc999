// bf16 attention dispatch: the tensor-core (mma.sync) split-KV kernel for
// decode tiles (one position) and few-position tiles.
#include "pa_attn_mma.cuh"

#ifndef PA_MMA_WARPS
#define PA_MMA_WARPS 4
#endif
#ifndef PA_MMA_STAGES
#define PA_MMA_STAGES 2
#endif
// head size 64: a K+V block is 4 KB, half the head-size-128 block
#ifndef PA_MMA_WARPS_D64
#define PA_MMA_WARPS_D64 PA_MMA_WARPS
#endif
#ifndef PA_MMA_STAGES_D64
#define PA_MMA_STAGES_D64 PA_MMA_STAGES
#endif

namespace pa {

namespace {
template <int D, int G>
cudaError_t dispatch_positions(const AttnParams& p, int positions, bool keys_as_m, int num_sms,
                               cudaStream_t stream, int* grid_only) {
  constexpr int NW = D == 64 ? PA_MMA_WARPS_D64 : PA_MMA_WARPS;
  constexpr int NS = D == 64 ? PA_MMA_STAGES_D64 : PA_MMA_STAGES;
  if (positions == 1)
    return keys_as_m ? launch_mma<D, G, 1, NW, NS, false, true>(p, num_sms, stream, grid_only)
                     : launch_mma<D, G, 1, NW, NS, false, false>(p, num_sms, stream, grid_only);
  return launch_mma<D, G, kSmallRows / G, NW, NS>(p, num_sms, stream, grid_only);
}

template <int D>
cudaError_t dispatch_group(const AttnParams& p, int group, int positions, bool keys_as_m,
                           int num_sms, cudaStream_t stream, int* grid_only) {
  switch (group) {
    case 1: return dispatch_positions<D, 1>(p, positions, keys_as_m, num_sms, stream, grid_only);
    case 2: return dispatch_positions<D, 2>(p, positions, keys_as_m, num_sms, stream, grid_only);
    case 4: return dispatch_positions<D, 4>(p, positions, keys_as_m, num_sms, stream, grid_only);
    case 8: return dispatch_positions<D, 8>(p, positions, keys_as_m, num_sms, stream, grid_only);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_attn_mma_bf16(const AttnParams& p, int head_size, int group, int positions,
                                 bool keys_as_m, int num_sms, cudaStream_t stream,
                                 int* grid_only) {
  switch (head_size) {
    case 64: return dispatch_group<64>(p, group, positions, keys_as_m, num_sms, stream, grid_only);
    case 128: return dispatch_group<128>(p, group, positions, keys_as_m, num_sms, stream, grid_only);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
