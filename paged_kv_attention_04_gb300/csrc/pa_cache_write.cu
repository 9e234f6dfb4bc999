// reshape_and_cache: scatter each new token's K and V row into its paged slot.
//
// "Inside vLLM: Anatomy of a High-Throughput LLM Inference System", section
// Run forward pass: slot_mapping is built with the inputs, and section Prefix
// Caching: the forward pass fills the allocated blocks with the new KVs.
//
// With the cache laid out [num_blocks][16][Hkv][D], slot s = block*16 + row
// names one contiguous row of Hkv*D elements, so the write is a row copy:
// every thread moves one 16-byte chunk of K and the same chunk of V with
// 128-bit loads and stores.  Bits are copied unchanged.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {
// Two floats -> two E4M3 codes (lo in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// 8 bf16 values (one 16-byte chunk) -> 8 E4M3 codes of x / scale.
__device__ __forceinline__ uint2 quantize8_e4m3(const uint4& w, float scale) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
  uint32_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    b[i] = e4m3x2(__fdiv_rn(bf16_lo(words[i]), scale), __fdiv_rn(bf16_hi(words[i]), scale));
  return make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}
}  // namespace

__global__ void __launch_bounds__(256) cache_write_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
    int num_tokens, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int row_chunks,
    long long num_slots, int32_t* status) {
  launch_dependents();  // a following plan kernel may start; it waits for this grid
  const long long total = static_cast<long long>(num_tokens) * row_chunks;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / row_chunks);
    const int c = static_cast<int>(i - static_cast<long long>(t) * row_chunks);
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= num_slots) {
      if (c == 0) flag_error(status, PA_DEV_SLOT_RANGE);
      continue;
    }
    const long long src = static_cast<long long>(t) * row_chunks + c;
    const long long dst = s * row_chunks + c;
    const uint4 kk = __ldg(k + src);
    const uint4 vv = __ldg(v + src);
    k_cache[dst] = kk;
    v_cache[dst] = vv;
  }
}

// FP8 (E4M3) variant: each thread turns one 16-byte chunk of bf16 K (and V)
// into 8 codes, code = E4M3(x / scale) with IEEE float32 division, round to
// nearest even, saturating (cvt.rn.satfinite).
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
    int num_tokens, uint2* __restrict__ k_cache, uint2* __restrict__ v_cache, int row_chunks,
    long long num_slots, float k_scale, float v_scale, int32_t* status) {
  launch_dependents();  // a following plan kernel may start; it waits for this grid
  const long long total = static_cast<long long>(num_tokens) * row_chunks;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / row_chunks);
    const int c = static_cast<int>(i - static_cast<long long>(t) * row_chunks);
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= num_slots) {
      if (c == 0) flag_error(status, PA_DEV_SLOT_RANGE);
      continue;
    }
    const long long src = static_cast<long long>(t) * row_chunks + c;
    const long long dst = s * row_chunks + c;
    k_cache[dst] = quantize8_e4m3(__ldg(k + src), k_scale);
    v_cache[dst] = quantize8_e4m3(__ldg(v + src), v_scale);
  }
}

cudaError_t launch_cache_write_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                                   int num_tokens, void* k_cache, void* v_cache, int row_bytes,
                                   long long num_slots, float k_scale, float v_scale,
                                   int32_t* status, cudaStream_t stream) {
  const int row_chunks = row_bytes / 16;  // bf16 input chunks per row
  const long long total = static_cast<long long>(num_tokens) * row_chunks;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 65535LL * 64) blocks = 65535LL * 64;
  cache_write_fp8_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, num_tokens,
      static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), row_chunks, num_slots, k_scale,
      v_scale, status);
  return cudaGetLastError();
}

cudaError_t launch_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                               int num_tokens, void* k_cache, void* v_cache, int row_bytes,
                               long long num_slots, int32_t* status, cudaStream_t stream) {
  const int row_chunks = row_bytes / 16;
  const long long total = static_cast<long long>(num_tokens) * row_chunks;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 65535LL * 64) blocks = 65535LL * 64;
  cache_write_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, num_tokens,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), row_chunks, num_slots, status);
  return cudaGetLastError();
}

}  // namespace pa
