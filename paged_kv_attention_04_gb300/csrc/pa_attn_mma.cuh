// bf16 paged attention for decode and few-token tiles: warp-level tensor-core
// products, a continuous per-warp KV stream, split-KV with a fused
// log-sum-exp merge.
//
// Decode is bound by HBM bandwidth ("Inside vLLM", section Scheduler).  On
// GB300 an SM must consume ~23 bytes of KV per clock to keep up with HBM;
// doing the grouped-query dot products on CUDA cores costs ~1400 warp
// instructions per 8 KB KV block (unpack, FMA, shuffles), which makes the
// kernel issue-bound.  The R = P x G query rows of a tile against a 16-token
// block are two tiny dense products (R x D by D x 16 and R x 16 by 16 x D),
// so each warp runs them as m16n8k16 bf16 MMAs with fp32 accumulation
// (rows padded to 16): ~32 MMAs and 16 ldmatrix per block.  The softmax
// stays on CUDA cores (fp32, base 2, quad shuffles).
//
// Work: units (request r, query tile m, KV split s, kv head g) fetched with
// an atomic counter.  A CTA has NW compute warps and one scheduler warp.
// The scheduler warp claims units two ahead, decodes them, copies the
// unit's block-table slice and stages the next unit's q rows, so the
// compute warps never wait on a dependent global load.  Compute warp w
// takes blocks w, w+NW, ... of a unit; its cp.async ring (NS stages of one
// K+V block, rows XOR-swizzled so ldmatrix is conflict-free) keeps issuing
// into the next unit's blocks while the current unit is finished, so the KV
// stream does not drain at unit boundaries.  Warps are joined through
// shared memory; a split unit writes (max, sum, acc) partials and the last
// split to finish merges them (atomic counter, no waiting).
//
// Causal limits: row j of a chunk of length L in a request of S tokens sits
// at position S - L + j ("Serving models at scale with vLLM", section
// Chunked prefill).  V rows past the last visible key are zero-filled so a
// masked (p = 0) key never meets unwritten (NaN) cache slots in the MMA.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "pa_device.cuh"
#include "pa_internal.h"

#ifndef PA_CLAIM_AHEAD
#define PA_CLAIM_AHEAD 0  // 1: the scheduler warp claims a unit one fetch early
#endif
#ifndef PA_SPARE_CLAIM
#define PA_SPARE_CLAIM 1  // 1: claim a second unit at the start only when units are plentiful
#endif
#ifndef PA_QK_SPLIT_ACC
#define PA_QK_SPLIT_ACC 0  // 1: two accumulator sets per score tile (shorter MMA chains)
#endif

// Prefetch each warp's next KV block into L2 while the cp.async ring streams
// the current one (1) or not (0).
#ifndef PA_L2_PREFETCH
#define PA_L2_PREFETCH 1
#endif
#ifndef PA_L2_PREFETCH_D64
#define PA_L2_PREFETCH_D64 0
#endif

namespace pa {

struct UnitMeta {
  int valid;
  int item, g, r, a, j0, npos, pos0, kv_hi, b0, b1, tile, nsplit, first;
  int bt[kMaxUnitBlocks];  // the unit's block-table slice
};

// What the scheduler warp keeps of a unit to finish it after the compute
// warps have moved on.
struct UnitTail {
  int valid, item, g, a, j0, npos, tile, nsplit, first;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Same with f16 inputs (used when the cache holds FP8 codes widened to f16).
__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two floats -> packed bf16 pair (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Transpose of an 8 x 8 matrix of 16-bit elements held one row pair per
// lane (lane l: row l / 4, columns 2 (l % 4), 2 (l % 4) + 1).
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(r) : "r"(x));
  return r;
}
// 2^x by the hardware approximation (ex2.approx.ftz: relative error about
// 2^-22, 0 for -inf), in place of the library exp2f: the softmax and the
// merges take 2^x of base-2 logits, and the shorter instruction sequence
// measured faster on the latency-bound FP8 and small decodes (FP8
// Llama-3-8B 139.3 -> 135.2 us, FP8 TinyLlama 24.6 -> 22.5 us).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// Two E4M3 codes (low byte first) -> two f16 values, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes16) {
  uint32_t r;
  const uint16_t c = static_cast<uint16_t>(codes16);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(c));
  return r;
}

// Four E4M3 codes (one 32-bit word, low byte first) -> two f16x2, exactly:
// codes 0-1 into lo, codes 2-3 into hi.  The word is unpacked into its 16-bit
// halves in PTX, which measured faster than shifting the high half down.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l16, h16;\n mov.b32 {l16, h16}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l16;\n cvt.rn.f16x2.e4m3x2 %1, h16;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// SW (decode tiles only, P = 1): the keys are the MMA's M dimension and the
// G <= 8 query rows its N; otherwise the query rows are M, padded to 16.
template <int D, int G, int P, int NW, int NS, bool F8, bool SW>
struct MmaCfg {
  static constexpr int kR = P * G;                 // real query rows (<= 16)
  static constexpr int kRowBytes = D * 2;          // a 16-bit tile row (bf16, or f16 from FP8)
  static constexpr int kChunks = kRowBytes / 16;   // 16-byte chunks per tile row
  static constexpr int kTileBytes = kBlockSize * kRowBytes;
  static constexpr int kCacheRowBytes = F8 ? D : D * 2;       // one cached row (token, head)
  static constexpr int kCacheChunks = kCacheRowBytes / 16;
  static constexpr int kRawTileBytes = F8 ? kBlockSize * D : 0;  // FP8 codes as copied
  // A ring stage holds one block's K and V as copied: swizzled 16-bit tiles, or
  // raw FP8 codes (16-byte chunks XOR-swizzled by row) read straight into MMA
  // fragments.
  static constexpr int kStageBytes = F8 ? 2 * kRawTileBytes : 2 * kTileBytes;
  static constexpr int kWarpRingBytes = NS * kStageBytes;
  static constexpr int kKSteps = D / 16;
  static constexpr int kNTiles = D / 8;
  static constexpr int kThreads = (NW + 1) * 32;
  static constexpr int kRingOff = 0;
  static constexpr int kRingBytes = NW * kWarpRingBytes;
  static constexpr int kQOff = kRingOff + kRingBytes;
  static constexpr int kQBytes = 2 * 16 * kRowBytes;
  static constexpr int kCombOff = kQOff + kQBytes;
  static constexpr int kCombBytes = 2 * NW * kR * D * 4;   // two units in flight
  static constexpr int kMlOff = kCombOff + kCombBytes;
  static constexpr int kMlBytes = 2 * NW * kR * 2 * 4;
  static constexpr int kMetaOff = (kMlOff + kMlBytes + 15) / 16 * 16;
  static constexpr int kSmemBytes = kMetaOff + 3 * static_cast<int>(sizeof(UnitMeta));
  // CTAs per SM that shared memory allows (228 KB per SM, 1 KB reserved per CTA):
  // two when they fit, three for FP8 keys-as-M tiles (their registers allow it)
  static constexpr int kFit = (228 * 1024) / (kSmemBytes + 1024 + 64);
  static constexpr int kMinCtas = (F8 && SW && kFit >= 3) ? 3 : (kFit >= 2 ? 2 : 1);
  static_assert(!SW || P == 1, "keys-as-M tiles are for decode (one position)");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA exceeds 227 KB");
  static_assert(kR <= 16, "at most 16 query rows per tile");
  static_assert(NS >= 2 && NS <= 8, "2 to 8 pipeline stages");
  static_assert(kChunks % 8 == 0, "rows must be a multiple of 128 bytes");
  static_assert((kBlockSize * kCacheChunks) % 32 == 0, "tile chunks must split over a warp");
};

// Swizzled byte offset of 16-byte chunk c of row t in a tile.
template <int RowBytes>
__device__ __forceinline__ uint32_t swz(int t, int c) {
  return static_cast<uint32_t>(t * RowBytes + ((c ^ (t & 7)) << 4));
}

template <int D, int G, int P, int NW, int NS, bool F8, bool SW>
__global__ void __launch_bounds__(MmaCfg<D, G, P, NW, NS, F8, SW>::kThreads,
                                  MmaCfg<D, G, P, NW, NS, F8, SW>::kMinCtas)
    attn_mma_kernel(const AttnParams p) {
  using C = MmaCfg<D, G, P, NW, NS, F8, SW>;
  constexpr int R = C::kR;
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool sched = warp == NW;
  const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
  UnitMeta* meta = reinterpret_cast<UnitMeta*>(smem + C::kMetaOff);
  float* comb = reinterpret_cast<float*>(smem + C::kCombOff);
  float* comb_ml = reinterpret_cast<float*>(smem + C::kMlOff);
  const uint32_t ring_u32 = smem_u32(smem + C::kRingOff) + warp * C::kWarpRingBytes;
  const uint32_t q_u32 = smem_u32(smem + C::kQOff);
  const unsigned char* kc = static_cast<const unsigned char*>(p.k_cache);
  const unsigned char* vc = static_cast<const unsigned char*>(p.v_cache);
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  wait_prior_grid();  // the plan's work lists
  const int n_units = __ldg(p.n_items) * Hkv;

  // ---- scheduler-warp helpers -------------------------------------------
  // Decode unit u (claimed earlier) into m: one precomputed record plus the
  // unit's block-table slice.
  auto fetch_unit = [&](UnitMeta& m, int u) {  // whole scheduler warp
    if (u >= n_units) {
      if (lane == 0) m.valid = 0;
      return;
    }
    const int k = u / Hkv;
    const int item = p.order ? __ldg(p.order + k) : k;
    const UnitRec* rec = p.recs + item;
    const int4 ra = __ldg(&rec->a), rb = __ldg(&rec->b), rc = __ldg(&rec->c);
    const int32_t* row = p.block_tables + static_cast<long long>(ra.x) * p.max_blocks_per_seq;
    for (int i = lane; i < ra.w - ra.z; i += 32) m.bt[i] = __ldg(row + ra.z + i);
    if (lane == 0) {
      m.valid = 1; m.item = item; m.g = u - k * Hkv; m.r = ra.x; m.a = rb.w; m.j0 = ra.y;
      m.npos = rc.x; m.pos0 = rc.y; m.kv_hi = rc.z; m.b0 = ra.z; m.b1 = ra.w;
      m.tile = rb.x; m.first = rb.y; m.nsplit = rb.z;
    }
  };
  auto claim = [&]() -> int {
    int u = 0;
    if (lane == 0) u = atomicAdd(p.next, 1);
    return __shfl_sync(0xffffffffu, u, 0);
  };
  // The CTA's first two units, decoded together so that their dependent
  // loads (dispatch slot, record, block-table slice) overlap.
  auto fetch_first_two = [&](int u0, int u1) {  // whole scheduler warp
    const bool v0 = u0 < n_units, v1 = u1 < n_units;
    const int k0 = u0 / Hkv, k1 = u1 / Hkv;
    int item0 = k0, item1 = k1;
    if (p.order) {
      if (v0) item0 = __ldg(p.order + k0);
      if (v1) item1 = __ldg(p.order + k1);
    }
    const int4 z = make_int4(0, 0, 0, 0);
    const int4 a0 = v0 ? __ldg(&p.recs[item0].a) : z, a1 = v1 ? __ldg(&p.recs[item1].a) : z;
    const int4 b0 = v0 ? __ldg(&p.recs[item0].b) : z, b1 = v1 ? __ldg(&p.recs[item1].b) : z;
    const int4 c0 = v0 ? __ldg(&p.recs[item0].c) : z, c1 = v1 ? __ldg(&p.recs[item1].c) : z;
    const int32_t* row0 = p.block_tables + static_cast<long long>(a0.x) * p.max_blocks_per_seq;
    const int32_t* row1 = p.block_tables + static_cast<long long>(a1.x) * p.max_blocks_per_seq;
    const int n0 = a0.w - a0.z, n1 = a1.w - a1.z;
    for (int i = lane; i < max(n0, n1); i += 32) {
      if (i < n0) meta[0].bt[i] = __ldg(row0 + a0.z + i);
      if (i < n1) meta[1].bt[i] = __ldg(row1 + a1.z + i);
    }
    if (lane == 0) {
      UnitMeta* m[2] = {&meta[0], &meta[1]};
      const int4 ra[2] = {a0, a1}, rb[2] = {b0, b1}, rc[2] = {c0, c1};
      const int us[2] = {u0, u1}, ks[2] = {k0, k1}, it[2] = {item0, item1};
      const bool vs[2] = {v0, v1};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        m[j]->valid = vs[j] ? 1 : 0;
        if (!vs[j]) continue;
        m[j]->item = it[j]; m[j]->g = us[j] - ks[j] * Hkv; m[j]->r = ra[j].x; m[j]->a = rb[j].w;
        m[j]->j0 = ra[j].y; m[j]->npos = rc[j].x; m[j]->pos0 = rc[j].y; m[j]->kv_hi = rc[j].z;
        m[j]->b0 = ra[j].z; m[j]->b1 = ra[j].w;
        m[j]->tile = rb[j].x; m[j]->first = rb[j].y; m[j]->nsplit = rb[j].z;
      }
    }
  };
  // q rows of unit m (row = position row/G, head row%G), loaded into registers
  // first and stored later, so the loads overlap other scheduler work.
  constexpr int kQPerLane = (R * C::kChunks + 31) / 32;
  auto load_q = [&](const UnitMeta& m, uint4 (&qv)[kQPerLane]) {
#pragma unroll
    for (int i = 0; i < kQPerLane; ++i) {
      const int idx = lane + 32 * i;
      const int row = idx / C::kChunks, c = idx - row * C::kChunks;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (m.valid && row < R) {
        const int jj = row / G, hh = row - jj * G;
        if (jj < m.npos) {
          const long long tok = m.a + m.j0 + jj;
          if constexpr (F8) {
            // f16, head dimension permuted to match the FP8 K fragments: logical
            // chunk c (k-step c/2, half c%2) holds bf16 pairs at words
            // (D/8)*t + 2*(c/2) + c%2 for t = 0..3 of the row (see the K loads)
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(q + (tok * Hq + m.g * G + hh) * D);
            const int wb = 2 * (c >> 1) + (c & 1);
            v = make_uint4(__ldg(qw + wb), __ldg(qw + (D / 8) + wb), __ldg(qw + 2 * (D / 8) + wb),
                           __ldg(qw + 3 * (D / 8) + wb));
          } else {
            v = __ldg(reinterpret_cast<const uint4*>(q + (tok * Hq + m.g * G + hh) * D) + c);
          }
        }
      }
      qv[i] = v;
    }
  };
  auto store_q = [&](const uint4 (&qv)[kQPerLane], int buf) {
#pragma unroll
    for (int i = 0; i < kQPerLane; ++i) {
      const int idx = lane + 32 * i;
      const int row = idx / C::kChunks, c = idx - row * C::kChunks;
      if (row < R) {
        uint4 v = qv[i];
        if constexpr (F8)
          v = make_uint4(pack_f16(bf16_lo(v.x), bf16_hi(v.x)), pack_f16(bf16_lo(v.y), bf16_hi(v.y)),
                         pack_f16(bf16_lo(v.z), bf16_hi(v.z)), pack_f16(bf16_lo(v.w), bf16_hi(v.w)));
        *reinterpret_cast<uint4*>(smem + C::kQOff + buf * 16 * C::kRowBytes +
                                  swz<C::kRowBytes>(row, c)) = v;
      }
    }
  };

  // scheduler-warp state kept in shared memory so it holds no registers in
  // the compute warps: the unit claimed for the next fetch, the unit to finish
  __shared__ int s_next_u;
  __shared__ UnitTail s_tail;
  if (sched) {
    // rows >= R of both q buffers stay zero for the whole kernel
    for (int idx = lane; idx < 2 * 16 * C::kChunks; idx += 32) {
      const int buf = idx / (16 * C::kChunks), rem = idx - buf * 16 * C::kChunks;
      const int row = rem / C::kChunks, c = rem - row * C::kChunks;
      if (row >= R)
        *reinterpret_cast<uint4*>(smem + C::kQOff + buf * 16 * C::kRowBytes +
                                  swz<C::kRowBytes>(row, c)) = make_uint4(0, 0, 0, 0);
    }
    // A second unit is claimed up front only if every CTA can still get one:
    // with fewer units than that (small steps), taking two would leave other
    // CTAs idle while this one works through both.
    int u0, u1;
    if (n_units >= 2 * static_cast<int>(gridDim.x)) {  // two units for every CTA: one claim
      int base = 0;
      if (lane == 0) base = atomicAdd(p.next, 2);
      u0 = __shfl_sync(0xffffffffu, base, 0);
      u1 = u0 + 1;
    } else {
      u0 = claim();
      u1 = (!PA_SPARE_CLAIM || u0 + static_cast<int>(gridDim.x) < n_units) ? claim() : n_units;
    }
    const int u2 = PA_CLAIM_AHEAD ? claim() : 0;
    if (lane == 0) {
      s_next_u = u2;
      s_tail.valid = 0;
    }
    fetch_first_two(u0, u1);
    __syncwarp();
    uint4 qv[kQPerLane];
    load_q(meta[0], qv);
    store_q(qv, 0);
  }
  __syncthreads();

  // ---- compute-warp stream state ----------------------------------------
  // The warp's KV stream is its share of unit k's blocks, then of unit k+1's.
  int iss_unit = 0, iss_i = 0;  // next block to issue: (unit sequence, index in warp share)
  int issued = 0, computed = 0;

  auto share = [&](const UnitMeta& m) -> int {
    const int n = m.b1 - m.b0 - warp;
    return (m.valid && n > 0) ? (n + NW - 1) / NW : 0;
  };
  // Issue the next block of the stream if it lies in unit `limit` or earlier.
  auto issue_one = [&](int limit) -> bool {
    while (iss_unit <= limit) {
      const UnitMeta& m = meta[iss_unit % 3];
      if (iss_i < share(m)) break;
      ++iss_unit;
      iss_i = 0;
    }
    if (iss_unit > limit) return false;
    const UnitMeta& m = meta[iss_unit % 3];
    const int bl = warp + iss_i * NW;  // block index within the unit
    const int b = m.b0 + bl;
    int phys = m.bt[bl];
    int kbytes = 16;
    if (phys < 0 || phys >= p.num_blocks) {
      if (lane == 0) flag_error(p.status, PA_DEV_BLOCK_RANGE);
      phys = 0;
      kbytes = 0;
    }
    const int valid_rows = min(kBlockSize, m.kv_hi - b * kBlockSize);
    const uint32_t st = ring_u32 + (issued % NS) * C::kStageBytes;
    const long long row_stride = static_cast<long long>(Hkv) * C::kCacheRowBytes;
    const long long base = static_cast<long long>(phys) * kBlockSize * row_stride +
                           static_cast<long long>(m.g) * C::kCacheRowBytes;
    const int c = lane % C::kCacheChunks;
#pragma unroll
    for (int k = 0; k < (kBlockSize * C::kCacheChunks) / 32; ++k) {
      const int t = lane / C::kCacheChunks + k * (32 / C::kCacheChunks);
      const long long off = base + t * row_stride + c * 16;
      const int vb = t < valid_rows ? kbytes : 0;
      if constexpr (F8) {  // raw codes, 16-byte chunks XOR-swizzled by row
        const uint32_t so = t * C::kCacheRowBytes + ((c ^ (t & (C::kCacheChunks - 1))) << 4);
        cp_async16(st + so, kc + off, vb);
        cp_async16(st + C::kRawTileBytes + so, vc + off, vb);
      } else {
        const uint32_t so = swz<C::kRowBytes>(t, c);
        cp_async16(st + so, kc + off, vb);
        cp_async16(st + C::kTileBytes + so, vc + off, vb);
      }
    }
    cp_async_commit();
    ++issued;
    ++iss_i;
    // Start the warp's next block of this unit towards L2 as well: one row per
    // lane (lanes 0-15 K, 16-31 V).  With the cp.async ring this keeps two
    // blocks per warp in flight from HBM without more shared memory (measured
    // on head size 128: +5.5 % decode bandwidth; head size 64 lost 8 %).
    if (PA_L2_PREFETCH && (D == 128 || PA_L2_PREFETCH_D64) && iss_i < share(m)) {
      const int nphys = m.bt[warp + iss_i * NW];
      if (nphys >= 0 && nphys < p.num_blocks) {
        const int t = lane & (kBlockSize - 1);
        const unsigned char* src = (lane < kBlockSize ? kc : vc) +
                                   static_cast<long long>(nphys) * kBlockSize * row_stride +
                                   static_cast<long long>(m.g) * C::kCacheRowBytes + t * row_stride;
#pragma unroll
        for (int l = 0; l < (C::kCacheRowBytes + 127) / 128; ++l)
          asm volatile("prefetch.global.L2 [%0];\n" ::"l"(src + l * 128));
      }
    }
    return true;
  };
  auto wait_for = [&](int idx) {  // block `idx` of the stream has landed
    const int newer = min(issued - idx - 1, NS - 1);  // groups allowed to stay in flight
    switch (newer) {
      case 7: cp_async_wait<7>(); break;
      case 6: cp_async_wait<6>(); break;
      case 5: cp_async_wait<5>(); break;
      case 4: cp_async_wait<4>(); break;
      case 3: cp_async_wait<3>(); break;
      case 2: cp_async_wait<2>(); break;
      case 1: cp_async_wait<1>(); break;
      default: cp_async_wait<0>(); break;
    }
    __syncwarp();
  };

  if (!sched) {
    for (int i = 0; i < NS - 1; ++i)
      if (!issue_one(1)) break;
  }

  // ---- scheduler warp: join the warps' states of a finished unit, write the
  // output or the split's partial, and merge the splits if it is the last.
  auto finish_unit = [&](const UnitTail& u, int buf) {
    const float* cb = comb + buf * NW * R * D;
    const float* cm = comb_ml + buf * NW * R * 2;
    const long long part_base = (static_cast<long long>(u.item) * Hkv + u.g) * R;
    for (int idx = lane; idx < R * D / 4; idx += 32) {
      const int row = (idx * 4) / D, d = idx * 4 - row * D;
      const int jj = row / G, hh = row - jj * G;
      if (jj >= u.npos) continue;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, cm[(w * R + row) * 2]);
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
      float den = 0.f;
      if (M != -CUDART_INF_F) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float f = ex2_approx(cm[(w * R + row) * 2] - M);
          const float4 c4 = *reinterpret_cast<const float4*>(cb + (w * R + row) * D + d);
          num.x = fmaf(c4.x, f, num.x); num.y = fmaf(c4.y, f, num.y);
          num.z = fmaf(c4.z, f, num.z); num.w = fmaf(c4.w, f, num.w);
          den = fmaf(cm[(w * R + row) * 2 + 1], f, den);
        }
      }
      if (u.nsplit == 1) {
        const long long tok = u.a + u.j0 + jj;
        const float inv = p.out_scale / den;
        *reinterpret_cast<uint2*>(out + (tok * Hq + u.g * G + hh) * D + d) =
            make_uint2(pack_bf16(num.x * inv, num.y * inv), pack_bf16(num.z * inv, num.w * inv));
      } else {
        *reinterpret_cast<float4*>(p.part_acc + (part_base + row) * D + d) = num;
        if (d == 0) *reinterpret_cast<float2*>(p.part_ml + (part_base + row) * 2) = make_float2(M, den);
      }
    }
    if (u.nsplit > 1) {
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(p.merge_cnt + u.tile * Hkv + u.g, 1) == u.nsplit - 1;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        // The partials sit in L2; each group of kMergeChunk splits is loaded
        // with independent loads before any is used, so a merge costs one
        // round trip per group instead of two per split.
        constexpr int kMergeChunk = 4;
#pragma unroll 2
        for (int idx = lane; idx < R * D / 4; idx += 32) {
          const int row = (idx * 4) / D, d = idx * 4 - row * D;
          const int jj = row / G, hh = row - jj * G;
          if (jj >= u.npos) continue;
          float M = -CUDART_INF_F, den = 0.f;
          float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int sp0 = 0; sp0 < u.nsplit; sp0 += kMergeChunk) {
            float2 ml[kMergeChunk];
            float4 a4[kMergeChunk];
#pragma unroll
            for (int j = 0; j < kMergeChunk; ++j) {
              ml[j] = make_float2(-CUDART_INF_F, 0.f);
              a4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (sp0 + j < u.nsplit) {
                const long long pb = (static_cast<long long>(u.first + sp0 + j) * Hkv + u.g) * R + row;
                ml[j] = __ldcg(reinterpret_cast<const float2*>(p.part_ml + pb * 2));
                a4[j] = __ldcg(reinterpret_cast<const float4*>(p.part_acc + pb * D + d));
              }
            }
            // a split with no visible key for this row holds (-inf, 0) and zeros
            float mc = M;
#pragma unroll
            for (int j = 0; j < kMergeChunk; ++j) mc = fmaxf(mc, ml[j].x);
            if (mc == -CUDART_INF_F) continue;
            if (mc > M) {  // rescale the running sums to the new maximum
              const float sc = ex2_approx(M - mc);  // 0 while nothing was visible
              num.x *= sc; num.y *= sc; num.z *= sc; num.w *= sc; den *= sc;
              M = mc;
            }
#pragma unroll
            for (int j = 0; j < kMergeChunk; ++j) {
              const float f = ex2_approx(ml[j].x - M);  // 0 for an empty split
              num.x = fmaf(a4[j].x, f, num.x); num.y = fmaf(a4[j].y, f, num.y);
              num.z = fmaf(a4[j].z, f, num.z); num.w = fmaf(a4[j].w, f, num.w);
              den = fmaf(ml[j].y, f, den);
            }
          }
          const long long tok = u.a + u.j0 + jj;
          const float inv = p.out_scale / den;
          *reinterpret_cast<uint2*>(out + (tok * Hq + u.g * G + hh) * D + d) =
              make_uint2(pack_bf16(num.x * inv, num.y * inv), pack_bf16(num.z * inv, num.w * inv));
        }
      }
    }
  };

  int k = 0;
  for (;; ++k) {
    const UnitMeta& cur = meta[k % 3];
    if (!cur.valid) break;
    if (sched) {
      // while the compute warps stream unit k: load unit k+1's q, finish unit
      // k-1, store the q rows, decode unit k+2 and claim the one after it
      uint4 qv[kQPerLane];
      load_q(meta[(k + 1) % 3], qv);
      const UnitTail tail = s_tail;
      if (tail.valid) finish_unit(tail, (k - 1) & 1);
      store_q(qv, (k + 1) & 1);
      // the stream ends at the first empty slot: claim nothing past it (a
      // unit claimed there would never be run)
      const int nu = meta[(k + 1) % 3].valid ? claim() : n_units;
      fetch_unit(meta[(k + 2) % 3], PA_CLAIM_AHEAD ? s_next_u : nu);
      __syncwarp();
      if (lane == 0) {
        s_next_u = nu;
        s_tail.valid = 1; s_tail.item = cur.item; s_tail.g = cur.g; s_tail.a = cur.a;
        s_tail.j0 = cur.j0; s_tail.npos = cur.npos; s_tail.tile = cur.tile;
        s_tail.nsplit = cur.nsplit; s_tail.first = cur.first;
      }
      __syncwarp();
    } else {
      // Every block of units < k has been issued and computed; move the issue
      // pointer off unit k-1, whose metadata slot the scheduler warp is now
      // overwriting with unit k+2.
      if (iss_unit < k) {
        iss_unit = k;
        iss_i = 0;
      }
      if constexpr (SW) {
        // Decode tile, keys as M: S^T = K Q^T (16 keys x 8 query rows) and
        // O^T += V^T P^T (16 head dims x 8 rows per m-tile): half the MMAs and
        // accumulators of a tile with the R <= 8 query rows padded to 16 as M.
        // Lane (g, c) = (lane / 4, lane % 4) holds S^T at keys g, g + 8 and
        // query rows 2c, 2c + 1, and O^T of m-tile mt at head dims
        // dim_of_m(mt, g), dim_of_m(mt, g + 8), rows 2c, 2c + 1.
        const int g = lane >> 2, c4 = lane & 3;
        const int r0 = 2 * c4, r1 = r0 + 1;  // this lane's query rows
        // q^T (B operand): b0 / b1 = dims 0-7 / 8-15 of k-step kk, q rows 0-7
        uint32_t qb[C::kKSteps][2];
        {
          const uint32_t qbuf = q_u32 + (k & 1) * 16 * C::kRowBytes;
#pragma unroll
          for (int kk = 0; kk < C::kKSteps; kk += 2)
            ldsm_x4(qbuf + swz<C::kRowBytes>(lane & 7, 2 * kk + (lane >> 3)), qb[kk][0], qb[kk][1],
                    qb[kk + 1][0], qb[kk + 1][1]);
        }
        float o[C::kKSteps][4];
#pragma unroll
        for (int j = 0; j < C::kKSteps; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
        const int nb = share(cur);
        for (int i = 0; i < nb; ++i) {
          issue_one(k + 1);
          wait_for(computed);
          const uint32_t st = ring_u32 + (computed % NS) * C::kStageBytes;
          const int tok0 = (cur.b0 + warp + i * NW) * kBlockSize;
          // S^T in two accumulators (even / odd k-steps): two shorter MMA chains
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (F8) {
            // K codes as A fragments: with the head dims permuted as on the q rows,
            // pi(kk, k) = (D/4)*((k%8)/2) + 4*kk + (k%2) + 2*(k/8), lane (g, c) needs
            // for k-step kk the 4 codes at (D/4)*c + 4*kk of keys g and g + 8
            uint32_t kw[2][D / 16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int t = g + 8 * h;
#pragma unroll
              for (int j = 0; j < D / 64; ++j) {
                const int cc = (D / 64) * c4 + j;
                uint4 v;
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                             : "r"(st + t * C::kCacheRowBytes + ((cc ^ (t & (C::kCacheChunks - 1))) << 4)));
                kw[h][4 * j] = v.x; kw[h][4 * j + 1] = v.y; kw[h][4 * j + 2] = v.z; kw[h][4 * j + 3] = v.w;
              }
            }
#pragma unroll
            for (int kk = 0; kk < C::kKSteps; ++kk) {
              uint32_t a[4];
              e4m3x4_to_f16x2x2(kw[0][kk], a[0], a[2]);
              e4m3x4_to_f16x2x2(kw[1][kk], a[1], a[3]);
              mma_f16((kk & 1) ? sb : sa, a, qb[kk][0], qb[kk][1]);
            }
          } else {
            // K rows as A fragments: matrices (keys 0-7 | 8-15) x (dims 0-7 | 8-15)
#pragma unroll
            for (int kk = 0; kk < C::kKSteps; ++kk) {
              uint32_t a[4];
              ldsm_x4(st + swz<C::kRowBytes>((lane & 7) + ((lane >> 3) & 1) * 8, 2 * kk + (lane >> 4)),
                      a[0], a[1], a[2], a[3]);
              mma_bf16((kk & 1) ? sb : sa, a, qb[kk][0], qb[kk][1]);
            }
          }
          // mask and online softmax (base 2): s[0] (key g, row r0), s[1] (key g, r1),
          // s[2] (key g + 8, r0), s[3] (key g + 8, r1); rows >= R are padding
          float s[4];
          {
            const int ka = tok0 + g, kb = ka + 8;
            const bool va = ka < cur.kv_hi && ka <= cur.pos0, vb = kb < cur.kv_hi && kb <= cur.pos0;
            const bool ra = r0 < R, rb = r1 < R;
            s[0] = (va && ra) ? (sa[0] + sb[0]) * p.scale_log2 : -CUDART_INF_F;
            s[1] = (va && rb) ? (sa[1] + sb[1]) * p.scale_log2 : -CUDART_INF_F;
            s[2] = (vb && ra) ? (sa[2] + sb[2]) * p.scale_log2 : -CUDART_INF_F;
            s[3] = (vb && rb) ? (sa[3] + sb[3]) * p.scale_log2 : -CUDART_INF_F;
          }
          float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
          for (int o8 = 4; o8 < 32; o8 <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o8));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o8));
          }
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          float corr0 = 1.f, corr1 = 1.f, pr[4];
          if (mn0 != -CUDART_INF_F) {
            corr0 = ex2_approx(m0 - mn0);
            pr[0] = ex2_approx(s[0] - mn0);
            pr[2] = ex2_approx(s[2] - mn0);
          } else {
            pr[0] = pr[2] = 0.f;
          }
          if (mn1 != -CUDART_INF_F) {
            corr1 = ex2_approx(m1 - mn1);
            pr[1] = ex2_approx(s[1] - mn1);
            pr[3] = ex2_approx(s[3] - mn1);
          } else {
            pr[1] = pr[3] = 0.f;
          }
          l0 = l0 * corr0 + (pr[0] + pr[2]);
          l1 = l1 * corr1 + (pr[1] + pr[3]);
          m0 = mn0;
          m1 = mn1;
          if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < C::kKSteps; ++mt) {
              o[mt][0] *= corr0; o[mt][1] *= corr1;
              o[mt][2] *= corr0; o[mt][3] *= corr1;
            }
          }
          // P^T as the B operand: an 8 x 8 transpose per half of the block's keys
          // takes (key g, rows 2c, 2c + 1) to (keys 2c, 2c + 1, row g)
          const uint32_t pb0 = movm_trans(F8 ? pack_f16(pr[0], pr[1]) : pack_bf16(pr[0], pr[1]));
          const uint32_t pb1 = movm_trans(F8 ? pack_f16(pr[2], pr[3]) : pack_bf16(pr[2], pr[3]));
          if constexpr (F8) {
            // V codes as A fragments of V^T: with the head dims of m-tile mt
            // permuted as dim_of_m(mt, m) = (D/8)*(m%8) + 2*mt + m/8, lane (g, c)
            // reads the D/8 codes at (D/8)*g of keys 2c, 2c+1, 2c+8, 2c+9 and
            // pairs two keys' codes per conversion
            const uint32_t vt = st + C::kRawTileBytes;
            uint32_t vw[4][D / 32];
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const int t = 2 * c4 + (i4 & 1) + 8 * (i4 >> 1);
              if constexpr (D == 128) {
                uint4 v;
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                             : "r"(vt + t * C::kCacheRowBytes + ((g ^ (t & 7)) << 4)));
                vw[i4][0] = v.x; vw[i4][1] = v.y; vw[i4][2] = v.z; vw[i4][3] = v.w;
              } else {
                uint2 v;
                asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];\n"
                             : "=r"(v.x), "=r"(v.y)
                             : "r"(vt + t * C::kCacheRowBytes + (((g >> 1) ^ (t & 3)) << 4) +
                                   ((g & 1) << 3)));
                vw[i4][0] = v.x; vw[i4][1] = v.y;
              }
            }
#pragma unroll
            for (int mt = 0; mt < C::kKSteps; ++mt) {
              const int w = mt >> 1;
              // dims 2mt and 2mt + 1 of two keys: one permute builds both pairs
              const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
              uint32_t a[4];
              e4m3x4_to_f16x2x2(__byte_perm(vw[0][w], vw[1][w], sel), a[0], a[1]);
              e4m3x4_to_f16x2x2(__byte_perm(vw[2][w], vw[3][w], sel), a[2], a[3]);
              mma_f16(o[mt], a, pb0, pb1);
            }
          } else {
            // V^T fragments by transposed ldmatrix: (keys 0-7 | 8-15) x (dims 0-7 | 8-15)
            const uint32_t vt = st + C::kTileBytes;
#pragma unroll
            for (int mt = 0; mt < C::kKSteps; ++mt) {
              uint32_t a[4];
              ldsm_x4_t(vt + swz<C::kRowBytes>((lane & 7) + (lane >> 4) * 8, 2 * mt + ((lane >> 3) & 1)),
                        a[0], a[1], a[2], a[3]);
              mma_bf16(o[mt], a, pb0, pb1);
            }
          }
          __syncwarp();
          ++computed;
        }
        // the warp's state for this unit -> shared memory (real rows only); row
        // sums over the 8 lanes (g) that share rows r0, r1
#pragma unroll
        for (int o8 = 4; o8 < 32; o8 <<= 1) {
          l0 += __shfl_xor_sync(0xffffffffu, l0, o8);
          l1 += __shfl_xor_sync(0xffffffffu, l1, o8);
        }
        float* cb = comb + (k & 1) * NW * R * D;
        float* cm = comb_ml + (k & 1) * NW * R * 2;
#pragma unroll
        for (int mt = 0; mt < C::kKSteps; ++mt)
#pragma unroll
          for (int hv = 0; hv < 2; ++hv) {
            const int dim = F8 ? (D / 8) * g + 2 * mt + hv : 16 * mt + g + 8 * hv;
            if (r0 < R) cb[(warp * R + r0) * D + dim] = o[mt][2 * hv];
            if (r1 < R) cb[(warp * R + r1) * D + dim] = o[mt][2 * hv + 1];
          }
        if (g == 0) {
          if (r0 < R) {
            cm[(warp * R + r0) * 2] = m0;
            cm[(warp * R + r0) * 2 + 1] = l0;
          }
          if (r1 < R) {
            cm[(warp * R + r1) * 2] = m1;
            cm[(warp * R + r1) * 2 + 1] = l1;
          }
        }
      } else {
      // q fragments (A operand, rows x D) for this unit
      uint32_t qa[C::kKSteps][4];
      {
        const uint32_t qb = q_u32 + (k & 1) * 16 * C::kRowBytes;
        const int mi = lane >> 3, rr = (lane & 7) + ((mi & 1) << 3);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          ldsm_x4(qb + swz<C::kRowBytes>(rr, 2 * kk + (mi >> 1)), qa[kk][0], qa[kk][1],
                  qa[kk][2], qa[kk][3]);
      }
      float o[C::kNTiles][4];
#pragma unroll
      for (int j = 0; j < C::kNTiles; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
      float mA = -CUDART_INF_F, mB = -CUDART_INF_F, lA = 0.f, lB = 0.f;
      const int rowA = lane >> 2, rowB = rowA + 8;
      const int nb = share(cur);
      for (int i = 0; i < nb; ++i) {
        issue_one(k + 1);
        wait_for(computed);
        const uint32_t st = ring_u32 + (computed % NS) * C::kStageBytes;

        const int tok0 = (cur.b0 + warp + i * NW) * kBlockSize;
        // S = Q K^T for the block's 16 tokens: two n-tiles of 8 tokens
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if constexpr (F8) {
          // K codes straight into B fragments.  With the head dimension permuted
          // as pi(kk, k) = (D/4)*((k%8)/2) + 4*kk + (k%2) + 2*(k/8) on Q and K alike,
          // lane (gid, tig) needs, for every k-step kk, the 4 codes at dims
          // (D/4)*tig + 4*kk .. +3 of tokens gid and gid + 8: one contiguous run of
          // D/4 bytes per token.
          const int gid = lane >> 2, tig = lane & 3;
          uint32_t kw[2][D / 16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int t = gid + 8 * h;
#pragma unroll
            for (int j = 0; j < D / 64; ++j) {
              const int c = (D / 64) * tig + j;
              uint4 v;
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                           : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                           : "r"(st + t * C::kCacheRowBytes + ((c ^ (t & (C::kCacheChunks - 1))) << 4)));
              kw[h][4 * j] = v.x; kw[h][4 * j + 1] = v.y; kw[h][4 * j + 2] = v.z; kw[h][4 * j + 3] = v.w;
            }
          }
          float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int kk = 0; kk < C::kKSteps; ++kk) {
            float* d0 = (PA_QK_SPLIT_ACC && (kk & 1)) ? s2[0] : s[0];
            float* d1 = (PA_QK_SPLIT_ACC && (kk & 1)) ? s2[1] : s[1];
            uint32_t b0[2], b1[2];
            e4m3x4_to_f16x2x2(kw[0][kk], b0[0], b0[1]);
            e4m3x4_to_f16x2x2(kw[1][kk], b1[0], b1[1]);
            mma_f16(d0, qa[kk], b0[0], b0[1]);
            mma_f16(d1, qa[kk], b1[0], b1[1]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            s[0][e] += s2[0][e];
            s[1][e] += s2[1][e];
          }
        } else {
          const int mi = lane >> 3;
          const int t = ((mi >> 1) << 3) + (lane & 7);
          float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int kk = 0; kk < C::kKSteps; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(st + swz<C::kRowBytes>(t, 2 * kk + (mi & 1)), b0, b1, b2, b3);
            float* d0 = (PA_QK_SPLIT_ACC && (kk & 1)) ? s2[0] : s[0];
            float* d1 = (PA_QK_SPLIT_ACC && (kk & 1)) ? s2[1] : s[1];
            mma_bf16(d0, qa[kk], b0, b1);
            mma_bf16(d1, qa[kk], b2, b3);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            s[0][e] += s2[0][e];
            s[1][e] += s2[1][e];
          }
        }
        // mask and online softmax (base 2); lane holds rows rowA (c0,c1) and rowB (c2,c3)
        float pA[4], pB[4];
        bool rescale;
        {
          float mx = -CUDART_INF_F;
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int tok = tok0 + j * 8 + ((lane & 3) << 1) + e;
              const int jj = rowA / G;
              const bool ok = rowA < R && jj < cur.npos && tok < cur.kv_hi && tok <= cur.pos0 + jj;
              s[j][e] = ok ? s[j][e] * p.scale_log2 : -CUDART_INF_F;
              mx = fmaxf(mx, s[j][e]);
            }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float mn = fmaxf(mA, mx);
          float corr = 1.f;
          if (mn != -CUDART_INF_F) {
            corr = ex2_approx(mA - mn);
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int e = 0; e < 2; ++e) pA[j * 2 + e] = ex2_approx(s[j][e] - mn);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) pA[e] = 0.f;
          }
          lA = lA * corr + (pA[0] + pA[1]) + (pA[2] + pA[3]);
          mA = mn;
          float corrB = 1.f;
          if constexpr (R > 8) {
            float mxb = -CUDART_INF_F;
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int tok = tok0 + j * 8 + ((lane & 3) << 1) + e;
                const int jj = rowB / G;
                const bool ok = rowB < R && jj < cur.npos && tok < cur.kv_hi && tok <= cur.pos0 + jj;
                s[j][2 + e] = ok ? s[j][2 + e] * p.scale_log2 : -CUDART_INF_F;
                mxb = fmaxf(mxb, s[j][2 + e]);
              }
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
            const float mnb = fmaxf(mB, mxb);
            if (mnb != -CUDART_INF_F) {
              corrB = ex2_approx(mB - mnb);
#pragma unroll
              for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) pB[j * 2 + e] = ex2_approx(s[j][2 + e] - mnb);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) pB[e] = 0.f;
            }
            lB = lB * corrB + (pB[0] + pB[1]) + (pB[2] + pB[3]);
            mB = mnb;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) pB[e] = 0.f;
          }
          rescale = __any_sync(0xffffffffu, corr != 1.f || corrB != 1.f);
          if (rescale) {
#pragma unroll
            for (int j = 0; j < C::kNTiles; ++j) {
              o[j][0] *= corr; o[j][1] *= corr;
              o[j][2] *= corrB; o[j][3] *= corrB;
            }
          }
        }
        // O += P V: P as the A operand (rows x 16 tokens), V via transposed ldmatrix
        uint32_t pa[4];
        if constexpr (F8) {
          pa[0] = pack_f16(pA[0], pA[1]);
          pa[1] = pack_f16(pB[0], pB[1]);
          pa[2] = pack_f16(pA[2], pA[3]);
          pa[3] = pack_f16(pB[2], pB[3]);
        } else {
          pa[0] = pack_bf16(pA[0], pA[1]);
          pa[1] = pack_bf16(pB[0], pB[1]);
          pa[2] = pack_bf16(pA[2], pA[3]);
          pa[3] = pack_bf16(pB[2], pB[3]);
        }
        if constexpr (F8) {
          // V codes straight into B fragments.  Output column n of n-tile nt is
          // head dim sigma(nt, n) = (D/8)*n + nt, so lane (gid, tig) needs dims
          // (D/8)*gid .. +D/8-1 of tokens 2tig, 2tig+1, 2tig+8, 2tig+9; byte pairs
          // from two tokens are interleaved and widened in one conversion.
          const int gid = lane >> 2, tig = lane & 3;
          const uint32_t vt = st + C::kRawTileBytes;
          uint32_t vw[4][D / 32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int t = 2 * tig + (i & 1) + 8 * (i >> 1);
            if constexpr (D == 128) {
              uint4 v;
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                           : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                           : "r"(vt + t * C::kCacheRowBytes + ((gid ^ (t & 7)) << 4)));
              vw[i][0] = v.x; vw[i][1] = v.y; vw[i][2] = v.z; vw[i][3] = v.w;
            } else {
              uint2 v;
              asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];\n"
                           : "=r"(v.x), "=r"(v.y)
                           : "r"(vt + t * C::kCacheRowBytes + (((gid >> 1) ^ (t & 3)) << 4) +
                                 ((gid & 1) << 3)));
              vw[i][0] = v.x; vw[i][1] = v.y;
            }
          }
#pragma unroll
          for (int w = 0; w < D / 32; ++w) {
            uint32_t l0[2], h0[2], l1[2], h1[2];
            e4m3x4_to_f16x2x2(__byte_perm(vw[0][w], vw[1][w], 0x5140), l0[0], l0[1]);
            e4m3x4_to_f16x2x2(__byte_perm(vw[0][w], vw[1][w], 0x7362), h0[0], h0[1]);
            e4m3x4_to_f16x2x2(__byte_perm(vw[2][w], vw[3][w], 0x5140), l1[0], l1[1]);
            e4m3x4_to_f16x2x2(__byte_perm(vw[2][w], vw[3][w], 0x7362), h1[0], h1[1]);
            mma_f16(o[4 * w + 0], pa, l0[0], l1[0]);
            mma_f16(o[4 * w + 1], pa, l0[1], l1[1]);
            mma_f16(o[4 * w + 2], pa, h0[0], h1[0]);
            mma_f16(o[4 * w + 3], pa, h0[1], h1[1]);
          }
        } else {
          const int mi = lane >> 3;
          const int t = ((mi & 1) << 3) + (lane & 7);
          const uint32_t vt = st + C::kTileBytes;
#pragma unroll
          for (int nt = 0; nt < C::kNTiles; nt += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vt + swz<C::kRowBytes>(t, nt + (mi >> 1)), b0, b1, b2, b3);
            mma_bf16(o[nt], pa, b0, b1);
            mma_bf16(o[nt + 1], pa, b2, b3);
          }
        }
        __syncwarp();
        ++computed;
      }
      // the warp's state for this unit -> shared memory (real rows only)
      float* cb = comb + (k & 1) * NW * R * D;
      float* cm = comb_ml + (k & 1) * NW * R * 2;
      lA += __shfl_xor_sync(0xffffffffu, lA, 1);
      lA += __shfl_xor_sync(0xffffffffu, lA, 2);
      lB += __shfl_xor_sync(0xffffffffu, lB, 1);
      lB += __shfl_xor_sync(0xffffffffu, lB, 2);
      // column n of n-tile j is head dim j*8 + n, or (D/8)*n + j on the FP8 path
      auto dim_of = [&](int j, int n) { return F8 ? (D / 8) * n + j : j * 8 + n; };
      if (rowA < R) {
#pragma unroll
        for (int j = 0; j < C::kNTiles; ++j) {
          if constexpr (F8) {
            cb[(warp * R + rowA) * D + dim_of(j, (lane & 3) << 1)] = o[j][0];
            cb[(warp * R + rowA) * D + dim_of(j, ((lane & 3) << 1) + 1)] = o[j][1];
          } else {
            *reinterpret_cast<float2*>(cb + (warp * R + rowA) * D + j * 8 + ((lane & 3) << 1)) =
                make_float2(o[j][0], o[j][1]);
          }
        }
        if ((lane & 3) == 0) {
          cm[(warp * R + rowA) * 2] = mA;
          cm[(warp * R + rowA) * 2 + 1] = lA;
        }
      }
      if constexpr (R > 8) {
        if (rowB < R) {
#pragma unroll
          for (int j = 0; j < C::kNTiles; ++j) {
            if constexpr (F8) {
              cb[(warp * R + rowB) * D + dim_of(j, (lane & 3) << 1)] = o[j][2];
              cb[(warp * R + rowB) * D + dim_of(j, ((lane & 3) << 1) + 1)] = o[j][3];
            } else {
              *reinterpret_cast<float2*>(cb + (warp * R + rowB) * D + j * 8 + ((lane & 3) << 1)) =
                  make_float2(o[j][2], o[j][3]);
            }
          }
          if ((lane & 3) == 0) {
            cm[(warp * R + rowB) * 2] = mB;
            cm[(warp * R + rowB) * 2 + 1] = lB;
          }
        }
      }
      }  // rows-as-M tile
    }
    __syncthreads();
  }
  if (sched) {
    const UnitTail tail = s_tail;
    if (tail.valid) finish_unit(tail, (k - 1) & 1);
  }
  cp_async_wait<0>();
}

// Launches the kernel, or with grid_only set only stores the grid size it
// would use (CTAs per SM by occupancy x SMs).
template <int D, int G, int P, int NW, int NS, bool F8 = false, bool SW = false>
cudaError_t launch_mma(const AttnParams& p, int num_sms, cudaStream_t stream,
                       int* grid_only = nullptr) {
  using C = MmaCfg<D, G, P, NW, NS, F8, SW>;
  static int ctas_per_sm[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (ctas_per_sm[dev] == 0) {
    e = cudaFuncSetAttribute(attn_mma_kernel<D, G, P, NW, NS, F8, SW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_mma_kernel<D, G, P, NW, NS, F8, SW>,
                                                      C::kThreads, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    ctas_per_sm[dev] = n > 0 ? n : 1;
  }
  if (grid_only) {
    *grid_only = num_sms * ctas_per_sm[dev];
    return cudaSuccess;
  }
  // right after the plan kernel the launch may overlap its tail (the kernel
  // waits for the plan before reading the work lists)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms * ctas_per_sm[dev]);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.after_plan ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_mma_kernel<D, G, P, NW, NS, F8, SW>, p);
}

}  // namespace pa
