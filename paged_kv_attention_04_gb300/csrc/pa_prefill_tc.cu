// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// A chunk of L new tokens of a request with S KV tokens: row j sits at
// position S - L + j and sees positions 0 .. S - L + j, its earlier chunks
// read back from the paged cache ("Serving models at scale with vLLM",
// section Chunked prefill; "Inside vLLM", section Chunked prefill).  With
// query length > 1 the two products are dense, so they run on tcgen05:
//
//   * a work unit is (request, kv head g, 128-row query tile); the rows are
//     128/G positions x the G q heads that share kv head g, so each K/V byte
//     staged serves 128 query rows;
//   * K and V tiles of 128 tokens (8 KV blocks, gathered through the block
//     table) are double-buffered by cp.async into 128-byte-swizzled shared
//     memory; Q, K and P are K-major operands, V an MN-major operand;
//   * S = Q K^T and O += P V are issued by one thread as
//     tcgen05.mma.kind::f16 (bf16 in, fp32 accumulate) into tensor memory;
//     completion is signalled through mbarriers (bounded waits);
//   * softmax: thread i owns query row i = TMEM lane i, reads its S row with
//     tcgen05.ld, masks causally, and writes P (bf16) back to shared memory.
//     The running maximum is only moved when a row's maximum grows by more
//     than 2^8 (base-2 logits), so O in tensor memory is rescaled rarely;
//     between moves p <= 2^8, well inside fp32 and bf16 range.
// Keys past the last visible position are zero-filled in V so masked
// probabilities never meet unwritten (NaN) cache slots.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kTileM = 128;              // query rows per unit
constexpr int kTileN = 128;              // KV tokens per tile
constexpr int kPfThreads = 128;          // one thread per query row
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr float kRescaleThreshold = 8.f; // base-2 logit growth that forces a rescale

template <int D>
struct PfCfg {
  static constexpr int kRegions = D / 64;                 // 128-byte column groups
  static constexpr int kTileBytes = kTileM * D * 2;       // Q, K or V tile
  static constexpr int kPBytes = kTileM * kTileN * 2;     // P tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTileBytes;        // 2 buffers
  static constexpr int kVOff = kKOff + 2 * kTileBytes;    // 2 buffers
  static constexpr int kPOff = kVOff + 2 * kTileBytes;    // 2 buffers
  static constexpr int kSmemBytes = kPOff + 2 * kPBytes + 1024;  // + alignment slack
  static constexpr int kTmemCols = 512;                   // S x 2 (256) + O (D <= 128)
  static constexpr int kChunks = D / 8;                   // 16-byte chunks per row
  static_assert(D == 64 || D == 128, "head size 64 or 128");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA exceeds 227 KB");
};

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile whose
// 64-element column groups are stacked regions of 128 rows x 128 bytes.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (kTileM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct UnitInfo {
  int r, g, a, j0, npos, pos0, kv_end;
};

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_tc_kernel(const AttnParams p) {
  using C = PfCfg<D>;
  constexpr int PM = kTileM / G;  // positions per unit
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t mbar[3];  // S done, O done, drain
  __shared__ uint32_t tmem_slot;
  __shared__ int s_unit;
  __shared__ UnitInfo s_info;

  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
  const unsigned char* kc = static_cast<const unsigned char*>(p.k_cache);
  const unsigned char* vc = static_cast<const unsigned char*>(p.v_cache);
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  const int n_units = __ldg(p.n_items) * Hkv;

  if (tid == 0) {
    mbar_init(smem_u32(&mbar[0]), 1);
    mbar_init(smem_u32(&mbar[1]), 1);
    mbar_init(smem_u32(&mbar[2]), 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tmem_s = tmem;        // S: two buffers, columns [0, 128) and [128, 256)
  const uint32_t tmem_o = tmem + 256;  // O: columns [256, 256 + D)
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  uint32_t ph_s = 0, ph_o = 0;
  bool aborted = false;

  // Load the K or V half (or both) of KV tile kt (tokens kt*128 ..) of unit u
  // into buffer buf.  Lanes take consecutive 16-byte chunks of a row (2 rows
  // per warp instruction for D=128); with the loop unrolled, the KV block of
  // every chunk a thread copies is known at compile time, so the tile's 8
  // block-table entries are read once, independently, before any copy.
  auto load_kv_part = [&](const UnitInfo& u, int kt, int buf, bool do_k, bool do_v) {
    const int32_t* bt_row = p.block_tables + static_cast<long long>(u.r) * p.max_blocks_per_seq;
    const long long row_stride = static_cast<long long>(Hkv) * D * 2;
    const uint32_t kdst = sbase + C::kKOff + buf * C::kTileBytes;
    const uint32_t vdst = sbase + C::kVOff + buf * C::kTileBytes;
    constexpr int kBlocks = kTileN / kBlockSize;
    long long base[kBlocks];
    int lim[kBlocks];  // tokens of block b (from its first) that exist; 0 for a bad id
#pragma unroll
    for (int b = 0; b < kBlocks; ++b) {
      const int tok0 = kt * kTileN + b * kBlockSize;
      base[b] = 0;
      lim[b] = 0;
      if (tok0 < u.kv_end) {
        const int phys = __ldg(bt_row + tok0 / kBlockSize);
        if (phys < 0 || phys >= p.num_blocks) {
          flag_error(p.status, PA_DEV_BLOCK_RANGE);
        } else {
          base[b] = static_cast<long long>(phys) * kBlockSize * row_stride +
                    static_cast<long long>(u.g) * D * 2;
          lim[b] = u.kv_end - tok0;
        }
      }
    }
    constexpr int kRowsPerPass = kPfThreads / C::kChunks;
    const int c = tid % C::kChunks;
#pragma unroll
    for (int k = 0; k < kTileN / kRowsPerPass; ++k) {
      const int tt = tid / C::kChunks + k * kRowsPerPass;
      const int b = (k * kRowsPerPass) / kBlockSize;  // compile-time (tt / 16)
      const int r = tt - b * kBlockSize;
      const int bytes = r < lim[b] ? 16 : 0;
      const long long off = bytes ? base[b] + r * row_stride + c * 16 : 0;
      if (do_k) cp_async16(kdst + sw128(tt, c), kc + off, bytes);
      if (do_v) cp_async16(vdst + sw128(tt, c), vc + off, bytes);
    }
  };
  auto load_kv = [&](const UnitInfo& u, int kt, int buf) { load_kv_part(u, kt, buf, true, true); };
  auto load_kv_k = [&](const UnitInfo& u, int kt, int buf) { load_kv_part(u, kt, buf, true, false); };
  auto load_kv_v = [&](const UnitInfo& u, int kt, int buf) { load_kv_part(u, kt, buf, false, true); };
  // S(kt) = Q K(kt)^T into TMEM S buffer sb (one thread).
  auto issue_s = [&](int kt, int sb) {
    const uint32_t qa = sbase + C::kQOff, kb = sbase + C::kKOff + (kt & 1) * C::kTileBytes;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t koff = (kk >> 2) * (kTileM * 128) + (kk & 3) * 32;
      tc_mma_f16(tmem_s + sb * kTileN, smem_desc_sw128(qa + koff, 16, 1024),
                 smem_desc_sw128(kb + koff, 16, 1024), idesc_bf16(kTileM, kTileN, 0), kk > 0);
    }
    tc_commit(smem_u32(&mbar[0]));
  };

  for (;;) {
    if (tid == 0) {
      const int unit = atomicAdd(p.next, 1);
      s_unit = unit;
      if (unit < n_units) {
        // last tile first: within a chunk later query tiles see more keys, and
        // later chunks of the step carry more prior context, so long units start first
        const int tile = __ldg(p.n_items) - 1 - unit / Hkv;
        const int4 tr = __ldg(p.items + tile);
        const int S = __ldg(p.seq_lens + tr.x);
        const int a = __ldg(p.qsl + tr.x);
        const int L = __ldg(p.qsl + tr.x + 1) - a;
        UnitInfo u;
        u.r = tr.x;
        u.g = unit % Hkv;
        u.a = a;
        u.j0 = tr.y * PM;
        u.npos = min(PM, L - u.j0);
        u.pos0 = S - L + u.j0;
        u.kv_end = u.pos0 + u.npos;
        s_info = u;
      }
    }
    __syncthreads();
    if (s_unit >= n_units || aborted) break;
    const UnitInfo u = s_info;
    const int n_kv = (u.kv_end + kTileN - 1) / kTileN;

    // Q tile: row i = (position i / G, head i % G); rows past the chunk are zero
    for (int idx = tid; idx < kTileM * C::kChunks; idx += kPfThreads) {
      const int row = idx / C::kChunks, c = idx - row * C::kChunks;
      const int jj = row / G, hh = row - jj * G;
      const bool ok = jj < u.npos;
      const long long tok = u.a + u.j0 + (ok ? jj : 0);
      cp_async16(sbase + C::kQOff + sw128(row, c),
                 q + (tok * Hq + u.g * G + hh) * D + c * 8, ok ? 16 : 0);
    }
    load_kv(u, 0, 0);
    cp_async_commit();
    if (n_kv > 1) load_kv_k(u, 1, 1);  // K of tile 1; its V follows one tile later
    cp_async_commit();

    // this thread's query row
    const int my_jj = tid / G;
    const bool row_ok = my_jj < u.npos;
    const int my_pos = u.pos0 + my_jj;
    float m_used = 0.f, l_sum = 0.f;

    // S(0) = Q K(0)^T
    cp_async_wait<1>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) issue_s(0, 0);

    // Per KV tile j: S(j+1) is issued before the softmax of tile j and PV(j)
    // is left in flight, so the tensor cores work while the threads do the
    // softmax.  Buffers: S in TMEM x2, K, V and P in shared memory x2.
    for (int kt = 0; kt < n_kv; ++kt) {
      const int buf = kt & 1;
      const bool ok_s = mbar_wait(smem_u32(&mbar[0]), ph_s, kWaitLimit);
      ph_s ^= 1;
      if (__syncthreads_or(!ok_s)) { aborted = true; break; }
      tc_fence_after();
      // PV(j-1) must be done before V(j+1) reuses its buffer (and before O is touched)
      if (kt > 0) {
        const bool ok_o = mbar_wait(smem_u32(&mbar[1]), ph_o, kWaitLimit);
        ph_o ^= 1;
        if (__syncthreads_or(!ok_o)) { aborted = true; break; }
        tc_fence_after();
      }
      // K(j+1) and V(j) have landed: issue S(j+1), then load V(j+1) and K(j+2)
      cp_async_wait<0>();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0 && kt + 1 < n_kv) issue_s(kt + 1, buf ^ 1);
      if (kt + 1 < n_kv) load_kv_v(u, kt + 1, buf ^ 1);
      if (kt + 2 < n_kv) load_kv_k(u, kt + 2, buf);
      cp_async_commit();

      // ---- softmax of this thread's row over the tile's 128 keys
      const int tok0 = kt * kTileN;
      uint32_t sr[kTileN];
#pragma unroll
      for (int c0 = 0; c0 < kTileN; c0 += 32) {
        uint32_t* dst = sr + c0;
        PA_TMEM_LD32(tmem_s + buf * kTileN + lane_off + c0, dst);
      }
      tmem_wait_ld();
      float mx4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int t = 0; t < kTileN; ++t) {
        const bool vis = row_ok && tok0 + t <= my_pos;
        const float x = vis ? __uint_as_float(sr[t]) * p.scale_log2 : -CUDART_INF_F;
        sr[t] = __float_as_uint(x);
        mx4[t & 3] = fmaxf(mx4[t & 3], x);
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      float factor = 1.f;
      if (row_ok) {
        if (kt == 0) {
          m_used = mx;  // position 0 is visible to every row, so mx is finite
        } else if (mx > m_used + kRescaleThreshold) {
          factor = exp2f(m_used - mx);
          l_sum *= factor;
          m_used = mx;
        }
      }
      // rescale O rows whose maximum moved (whole warp takes part in tcgen05.ld/st);
      // PV(j-1) is complete, so O is stable
      if (kt > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          PA_TMEM_LD32(tmem_o + lane_off + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * factor);
          PA_TMEM_ST32(tmem_o + lane_off + c0, o);
        }
        tmem_wait_st();
      }
      // P = exp2(x - m_used) as bf16, K-major rows of 128 keys, into P buffer j%2
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t prow = sbase + C::kPOff + buf * C::kPBytes;
#pragma unroll
      for (int c = 0; c < kTileN / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = exp2f(__uint_as_float(sr[c * 8 + 2 * e]) - m_used);
          const float p1 = exp2f(__uint_as_float(sr[c * 8 + 2 * e + 1]) - m_used);
          ps4[e] += p0 + p1;
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(w[e]) : "f"(p1), "f"(p0));
        }
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + sw128(tid, c)),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
      }
      l_sum += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
        const uint32_t pa = sbase + C::kPOff + buf * C::kPBytes;
        const uint32_t vb = sbase + C::kVOff + buf * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          tc_mma_f16(tmem_o, smem_desc_sw128(pa + (kk >> 2) * (kTileM * 128) + (kk & 3) * 32, 16, 1024),
                     smem_desc_sw128(vb + kk * 2048, kTileM * 128, 1024), idesc_bf16(kTileM, D, 1),
                     (kt > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&mbar[1]));
      }
    }
    if (!aborted) {  // the last PV
      const bool ok_o = mbar_wait(smem_u32(&mbar[1]), ph_o, kWaitLimit);
      ph_o ^= 1;
      if (__syncthreads_or(!ok_o)) aborted = true;
      tc_fence_after();
    }
    if (aborted) break;

    // ---- O / l -> out
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t o[32];
      PA_TMEM_LD32(tmem_o + lane_off + c0, o);
      tmem_wait_ld();
      if (row_ok) {
        const float inv = 1.f / l_sum;
        const long long tok = u.a + u.j0 + my_jj;
        uint4* dst = reinterpret_cast<uint4*>(out + (tok * Hq + u.g * G + (tid - my_jj * G)) * D + c0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 v;
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(v.x) : "f"(__uint_as_float(o[8 * j + 1]) * inv), "f"(__uint_as_float(o[8 * j]) * inv));
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(v.y) : "f"(__uint_as_float(o[8 * j + 3]) * inv), "f"(__uint_as_float(o[8 * j + 2]) * inv));
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(v.z) : "f"(__uint_as_float(o[8 * j + 5]) * inv), "f"(__uint_as_float(o[8 * j + 4]) * inv));
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(v.w) : "f"(__uint_as_float(o[8 * j + 7]) * inv), "f"(__uint_as_float(o[8 * j + 6]) * inv));
          dst[j] = v;
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  cp_async_wait<0>();
  if (aborted) {
    if (tid == 0) {
      flag_error(p.status, PA_DEV_TIMEOUT);
      tc_commit(smem_u32(&mbar[2]));  // completes once every MMA issued so far is done
    }
    mbar_wait(smem_u32(&mbar[2]), 0, kWaitLimit);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

namespace {
template <int D, int G>
cudaError_t launch_pf(const AttnParams& p, int num_sms, cudaStream_t stream) {
  using C = PfCfg<D>;
  static int ctas_per_sm[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (ctas_per_sm[dev] == 0) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_tc_kernel<D, G>, kPfThreads,
                                                      C::kSmemBytes);
    if (e != cudaSuccess) return e;
    // each CTA holds 256 TMEM columns; two CTAs fill an SM's 512
    ctas_per_sm[dev] = n < 1 ? 1 : (n > 2 ? 2 : n);
  }
  prefill_tc_kernel<D, G><<<num_sms * ctas_per_sm[dev], kPfThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefill_tc(const AttnParams& p, int head_size, int group, int num_sms,
                              cudaStream_t stream) {
  if (head_size == 128) {
    switch (group) {
      case 1: return launch_pf<128, 1>(p, num_sms, stream);
      case 2: return launch_pf<128, 2>(p, num_sms, stream);
      case 4: return launch_pf<128, 4>(p, num_sms, stream);
      case 8: return launch_pf<128, 8>(p, num_sms, stream);
    }
  } else if (head_size == 64) {
    switch (group) {
      case 1: return launch_pf<64, 1>(p, num_sms, stream);
      case 2: return launch_pf<64, 2>(p, num_sms, stream);
      case 4: return launch_pf<64, 4>(p, num_sms, stream);
      case 8: return launch_pf<64, 8>(p, num_sms, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
