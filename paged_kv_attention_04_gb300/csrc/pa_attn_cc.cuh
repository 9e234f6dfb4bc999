// CUDA-core paged attention with split-KV and a fused log-sum-exp merge.
//
// Decode is bound by HBM bandwidth ("Inside vLLM", section Scheduler: a decode
// step must load all cached KV to produce one token), so this kernel is built
// to stream KV blocks at full bandwidth and keep arithmetic off the critical
// path:
//   * one work unit = (request r, query tile m, KV split s, kv head g); units
//     are fetched dynamically with one atomic per unit so the SMs stay evenly
//     loaded under skewed lengths;
//   * the tile's rows are P query positions x G grouped q heads; all R = P*G
//     rows share every K/V byte read (the GQA group shares the KV head);
//   * each warp streams its own 16-token blocks through a private
//     cp.async ring of 16-byte copies (K rows swizzled in shared memory so the
//     score loop is bank-conflict free), so no CTA barrier sits in the loop;
//   * scores: lane (t, half) owns token t and half of the head dimension; one
//     shuffle joins the halves.  Online softmax in base 2 with warp shuffles.
//     P.V: each lane owns D/32 output dimensions;
//   * warps are joined through shared memory at the end of a unit; a split
//     tile writes its (max, sum, acc) partial and the last split to arrive
//     merges all partials (atomic counter, no waiting).
//
// The block table is read with the block index of the logical position
// ("Serving models at scale with vLLM", section PagedAttention); causal
// limits follow "Serving models at scale with vLLM", section Chunked prefill:
// row j of a q_len-L chunk of a request with S tokens sits at S - L + j.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

template <typename T, int D, int G, int P>
struct CcCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kR = P * G;                       // rows per tile
  static constexpr int kRP = (kR + 3) / 4 * 4;           // padded row count
  static constexpr int kRowBytes = D * Elem<T>::kBytes;  // one token, one head
  static constexpr int kChunks = kRowBytes / 16;         // 16-byte chunks per row
  static constexpr int kEpc = Chunk<T>::kElems;          // elements per chunk
  static constexpr int kHalfChunks = kChunks / 2;
  static constexpr int kTileBytes = kBlockSize * kRowBytes;   // K (or V) of one block
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = kStageBytes >= 16384 ? 2 : 3;
  static constexpr int kDpl = D / 32;                    // output dims per lane
  static constexpr int kQStride = D / 2 + 4;             // floats per q half-row
  // shared memory layout (bytes)
  static constexpr int kRingOff = 0;
  static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
  static constexpr int kQOff = kRingOff + kRingBytes;
  static constexpr int kQBytes = kR * 2 * kQStride * 4;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kPBytes = kWarps * kBlockSize * kRP * 4;
  static constexpr int kCombAccOff = kPOff + kPBytes;
  static constexpr int kCombAccBytes = kWarps * kR * D * 4;
  static constexpr int kCombMlOff = kCombAccOff + kCombAccBytes;
  static constexpr int kCombMlBytes = kWarps * kR * 2 * 4;
  static constexpr int kSmemBytes = kCombMlOff + kCombMlBytes;
  static_assert(kChunks >= 8 && kChunks % 8 == 0, "row must be a multiple of 128 bytes");
  static_assert((kBlockSize * kChunks) % 32 == 0, "tile chunks must split over a warp");
  static_assert(D % 32 == 0, "head size must be a multiple of 32");
};

template <typename T, int D, int G, int P>
__global__ void __launch_bounds__(CcCfg<T, D, G, P>::kThreads)
    attn_cc_kernel(const AttnParams p) {
  using C = CcCfg<T, D, G, P>;
  constexpr int R = C::kR;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_unit;
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int t_lane = lane & 15;   // token owned in the score loop
  const int half = lane >> 4;     // half of the head dimension owned
  const int Hkv = p.num_kv_heads;
  const int Hq = p.num_q_heads;
  const int n_units = __ldg(p.n_items) * Hkv;

  float* q_s = reinterpret_cast<float*>(smem + C::kQOff);
  float* p_s = reinterpret_cast<float*>(smem + C::kPOff) + warp * kBlockSize * C::kRP;
  float* comb_acc = reinterpret_cast<float*>(smem + C::kCombAccOff);
  float* comb_ml = reinterpret_cast<float*>(smem + C::kCombMlOff);
  unsigned char* ring = smem + C::kRingOff + warp * C::kStages * C::kStageBytes;
  const uint32_t ring_u32 = smem_u32(ring);

  const unsigned char* kc = static_cast<const unsigned char*>(p.k_cache);
  const unsigned char* vc = static_cast<const unsigned char*>(p.v_cache);
  const T* q = static_cast<const T*>(p.q);
  T* out = static_cast<T*>(p.out);

  for (;;) {
    if (tid == 0) s_unit = atomicAdd(p.next, 1);
    __syncthreads();
    const int unit = s_unit;
    if (unit >= n_units) break;
    const int k = unit / Hkv;
    const int item = p.order ? __ldg(p.order + k) : k;
    const int g = unit - k * Hkv;
    const int4 it = __ldg(p.items + item);
    const int r = it.x, m = it.y, tile = it.w;
    const int4 tinfo = __ldg(p.tiles + tile);
    const int nsplit = tinfo.y;
    const int S = __ldg(p.seq_lens + r);
    const int a = __ldg(p.qsl + r);
    const int L = __ldg(p.qsl + r + 1) - a;
    const int j0 = m * P;
    const int npos = min(P, L - j0);             // valid positions in the tile
    const int pos0 = S - L + j0;                 // position of tile row 0
    const int kv_end = pos0 + npos;              // one past the last visible key
    const int nblk = (kv_end + kBlockSize - 1) / kBlockSize;
    const int b0 = it.z;
    const int b1 = min(b0 + tinfo.z, nblk);
    const int kv_hi = min(b1 * kBlockSize, kv_end);
    const int32_t* bt_row = p.block_tables + static_cast<long long>(r) * p.max_blocks_per_seq;

    // q rows of the tile, as fp32, split into two half-rows per row.
    for (int idx = tid; idx < R * D; idx += C::kThreads) {
      const int row = idx / D, d = idx - row * D;
      const int jj = row / G, hh = row - jj * G;
      float val = 0.f;
      if (jj < npos) {
        const long long tok = a + j0 + jj;
        val = Elem<T>::to_float(q[(tok * Hq + g * G + hh) * D + d]);
      }
      q_s[(row * 2 + d / (D / 2)) * C::kQStride + (d % (D / 2))] = val;
    }
    __syncthreads();

    // ---- per-warp pipeline over blocks b0+warp, b0+warp+W, ...
    const int nb_w = (b1 - b0 - warp + C::kWarps - 1) / C::kWarps > 0
                         ? (b1 - b0 - warp + C::kWarps - 1) / C::kWarps : 0;
    float m_run[R], l_run[R], acc[R][C::kDpl];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      m_run[i] = -CUDART_INF_F;
      l_run[i] = 0.f;
#pragma unroll
      for (int d = 0; d < C::kDpl; ++d) acc[i][d] = 0.f;
    }

    auto issue = [&](int i) {
      const int b = b0 + warp + i * C::kWarps;
      int phys = __ldg(bt_row + b);
      int bytes = 16;
      if (phys < 0 || phys >= p.num_blocks) {
        if (lane == 0) flag_error(p.status, PA_DEV_BLOCK_RANGE);
        phys = 0;
        bytes = 0;
      }
      const uint32_t st = ring_u32 + (i % C::kStages) * C::kStageBytes;
      const long long row0 = (static_cast<long long>(phys) * kBlockSize * Hkv + g) * C::kRowBytes;
      const long long row_stride = static_cast<long long>(Hkv) * C::kRowBytes;
#pragma unroll
      for (int k = 0; k < (kBlockSize * C::kChunks) / 32; ++k) {
        const int idx = lane + 32 * k;
        const int t = idx / C::kChunks, c = idx % C::kChunks;
        const long long off = row0 + t * row_stride + c * 16;
        cp_async16(st + t * C::kRowBytes + ((c ^ (t & 7)) * 16), kc + off, bytes);
        cp_async16(st + C::kTileBytes + t * C::kRowBytes + c * 16, vc + off, bytes);
      }
    };

#pragma unroll
    for (int i = 0; i < C::kStages - 1; ++i) {
      if (i < nb_w) issue(i);
      cp_async_commit();
    }
    for (int i = 0; i < nb_w; ++i) {
      if (i + C::kStages - 1 < nb_w) issue(i + C::kStages - 1);
      cp_async_commit();
      cp_async_wait<C::kStages - 1>();
      __syncwarp();
      const unsigned char* st = ring + (i % C::kStages) * C::kStageBytes;
      const int b = b0 + warp + i * C::kWarps;
      const int tok0 = b * kBlockSize;

      // scores for token t_lane, half `half` of the dimension
      float sc[R];
#pragma unroll
      for (int row = 0; row < R; ++row) sc[row] = 0.f;
      const unsigned char* krow = st + t_lane * C::kRowBytes;
#pragma unroll
      for (int i2 = 0; i2 < C::kHalfChunks; ++i2) {
        const int c = half * C::kHalfChunks + i2;
        const uint4 raw = *reinterpret_cast<const uint4*>(krow + ((c ^ (t_lane & 7)) * 16));
        float kf[C::kEpc];
        Chunk<T>::unpack(raw, kf);
#pragma unroll
        for (int row = 0; row < R; ++row) {
          const float* qh = q_s + (row * 2 + half) * C::kQStride + i2 * C::kEpc;
#pragma unroll
          for (int e = 0; e < C::kEpc; e += 4) {
            const float4 q4 = *reinterpret_cast<const float4*>(qh + e);
            sc[row] = fmaf(q4.x, kf[e], sc[row]);
            sc[row] = fmaf(q4.y, kf[e + 1], sc[row]);
            sc[row] = fmaf(q4.z, kf[e + 2], sc[row]);
            sc[row] = fmaf(q4.w, kf[e + 3], sc[row]);
          }
        }
      }
      const int tok = tok0 + t_lane;
#pragma unroll
      for (int row = 0; row < R; ++row) {
        sc[row] += __shfl_xor_sync(0xffffffffu, sc[row], 16);
        const int jj = row / G;
        const bool ok = tok < kv_hi && tok <= pos0 + jj && jj < npos;
        sc[row] = ok ? sc[row] * p.scale_log2 : -CUDART_INF_F;
      }
      // online softmax over the block's 16 tokens
#pragma unroll
      for (int row = 0; row < R; ++row) {
        float bm = sc[row];
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        const float m_new = fmaxf(m_run[row], bm);
        float pr = 0.f, corr = 1.f;
        if (m_new != -CUDART_INF_F) {
          pr = exp2f(sc[row] - m_new);
          corr = exp2f(m_run[row] - m_new);
        }
        float ps = pr;
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 4);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        l_run[row] = l_run[row] * corr + ps;
        m_run[row] = m_new;
#pragma unroll
        for (int d = 0; d < C::kDpl; ++d) acc[row][d] *= corr;
        if (half == 0) p_s[t_lane * C::kRP + row] = pr;
      }
      __syncwarp();
      // P.V over the valid tokens of the block
      const unsigned char* vtile = st + C::kTileBytes;
      const int ntok = min(kBlockSize, kv_hi - tok0);
      for (int tt = 0; tt < ntok; ++tt) {
        float vf[C::kDpl];
        const unsigned char* vrow = vtile + tt * C::kRowBytes + lane * C::kDpl * Elem<T>::kBytes;
        if constexpr (Elem<T>::kBytes == 2) {
          if constexpr (C::kDpl == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(vrow);
            vf[0] = bf16_lo(w.x); vf[1] = bf16_hi(w.x); vf[2] = bf16_lo(w.y); vf[3] = bf16_hi(w.y);
          } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow);
            vf[0] = bf16_lo(w); vf[1] = bf16_hi(w);
          }
        } else {
          if constexpr (C::kDpl == 4) {
            const float4 w = *reinterpret_cast<const float4*>(vrow);
            vf[0] = w.x; vf[1] = w.y; vf[2] = w.z; vf[3] = w.w;
          } else {
            const float2 w = *reinterpret_cast<const float2*>(vrow);
            vf[0] = w.x; vf[1] = w.y;
          }
        }
        const float* prow = p_s + tt * C::kRP;
#pragma unroll
        for (int row = 0; row < R; ++row) {
          const float pr = prow[row];
#pragma unroll
          for (int d = 0; d < C::kDpl; ++d) acc[row][d] = fmaf(pr, vf[d], acc[row][d]);
        }
      }
      __syncwarp();
    }
    cp_async_wait<0>();

    // ---- join the warps
#pragma unroll
    for (int row = 0; row < R; ++row) {
#pragma unroll
      for (int d = 0; d < C::kDpl; ++d)
        comb_acc[(warp * R + row) * D + lane * C::kDpl + d] = acc[row][d];
      if (lane == 0) {
        comb_ml[(warp * R + row) * 2] = m_run[row];
        comb_ml[(warp * R + row) * 2 + 1] = l_run[row];
      }
    }
    __syncthreads();
    const long long part_base = (static_cast<long long>(item) * Hkv + g) * R;
    for (int idx = tid; idx < R * D; idx += C::kThreads) {
      const int row = idx / D, d = idx - row * D;
      const int jj = row / G, hh = row - jj * G;
      if (jj >= npos) continue;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, comb_ml[(w * R + row) * 2]);
      float num = 0.f, den = 0.f;
      if (M != -CUDART_INF_F) {
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) {
          const float f = exp2f(comb_ml[(w * R + row) * 2] - M);
          num = fmaf(comb_acc[(w * R + row) * D + d], f, num);
          den = fmaf(comb_ml[(w * R + row) * 2 + 1], f, den);
        }
      }
      if (nsplit == 1) {
        const long long tok = a + j0 + jj;
        out[(tok * Hq + g * G + hh) * D + d] = Elem<T>::from_float(num / den);
      } else {
        p.part_acc[(part_base + row) * D + d] = num;
        if (d == 0) {
          p.part_ml[(part_base + row) * 2] = M;
          p.part_ml[(part_base + row) * 2 + 1] = den;
        }
      }
    }
    if (nsplit > 1) {
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int prev = atomicAdd(p.merge_cnt + tile * Hkv + g, 1);
        s_last = (prev == nsplit - 1);
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        const int first = tinfo.x;
        for (int idx = tid; idx < R * D; idx += C::kThreads) {
          const int row = idx / D, d = idx - row * D;
          const int jj = row / G, hh = row - jj * G;
          if (jj >= npos) continue;
          float M = -CUDART_INF_F;
          for (int k = 0; k < nsplit; ++k) {
            const long long pb = (static_cast<long long>(first + k) * Hkv + g) * R + row;
            M = fmaxf(M, __ldcg(p.part_ml + pb * 2));
          }
          float num = 0.f, den = 0.f;
          for (int k = 0; k < nsplit; ++k) {
            const long long pb = (static_cast<long long>(first + k) * Hkv + g) * R + row;
            const float f = exp2f(__ldcg(p.part_ml + pb * 2) - M);
            num = fmaf(__ldcg(p.part_acc + pb * D + d), f, num);
            den = fmaf(__ldcg(p.part_ml + pb * 2 + 1), f, den);
          }
          const long long tok = a + j0 + jj;
          out[(tok * Hq + g * G + hh) * D + d] = Elem<T>::from_float(num / den);
        }
      }
    }
    __syncthreads();
  }
}

// Occupancy and shared-memory opt-in, computed once per device.
template <typename T, int D, int G, int P>
cudaError_t launch_cc(const AttnParams& p, int num_sms, cudaStream_t stream,
                      int* grid_only = nullptr) {
  using C = CcCfg<T, D, G, P>;
  static int ctas_per_sm[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (ctas_per_sm[dev] == 0) {
    e = cudaFuncSetAttribute(attn_cc_kernel<T, D, G, P>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_cc_kernel<T, D, G, P>, C::kThreads,
                                                      C::kSmemBytes);
    if (e != cudaSuccess) return e;
    ctas_per_sm[dev] = n > 0 ? n : 1;
  }
  const int grid = num_sms * ctas_per_sm[dev];
  if (grid_only) {
    *grid_only = grid;
    return cudaSuccess;
  }
  attn_cc_kernel<T, D, G, P><<<grid, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t dispatch_cc_group(const AttnParams& p, int group, int positions, int num_sms,
                              cudaStream_t stream, int* grid_only) {
  const bool dec = positions == 1;
  switch (group) {
    case 1: return dec ? launch_cc<T, D, 1, 1>(p, num_sms, stream, grid_only)
                       : launch_cc<T, D, 1, kSmallRows / 1>(p, num_sms, stream, grid_only);
    case 2: return dec ? launch_cc<T, D, 2, 1>(p, num_sms, stream, grid_only)
                       : launch_cc<T, D, 2, kSmallRows / 2>(p, num_sms, stream, grid_only);
    case 4: return dec ? launch_cc<T, D, 4, 1>(p, num_sms, stream, grid_only)
                       : launch_cc<T, D, 4, kSmallRows / 4>(p, num_sms, stream, grid_only);
    case 8: return dec ? launch_cc<T, D, 8, 1>(p, num_sms, stream, grid_only)
                       : launch_cc<T, D, 8, kSmallRows / 8>(p, num_sms, stream, grid_only);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t dispatch_cc(const AttnParams& p, int head_size, int group, int positions, int num_sms,
                        cudaStream_t stream, int* grid_only) {
  switch (head_size) {
    case 64: return dispatch_cc_group<T, 64>(p, group, positions, num_sms, stream, grid_only);
    case 128: return dispatch_cc_group<T, 128>(p, group, positions, num_sms, stream, grid_only);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
