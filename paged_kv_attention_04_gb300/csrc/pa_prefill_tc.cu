// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05),
// warp-specialised.
//
// A chunk of L new tokens of a request with S KV tokens: row j sits at
// position S - L + j and sees positions 0 .. S - L + j, its earlier chunks
// read back from the paged cache ("Serving models at scale with vLLM",
// section Chunked prefill; "Inside vLLM", section Chunked prefill).  With
// query length > 1 the two products are dense, so they run on tcgen05.
//
// Work unit: (request, kv head g, 128-row query tile); the rows are 128/G
// positions x the G q heads that share kv head g, so every K/V byte staged
// serves 128 query rows.  Units are fetched from a counter, longest first.
// One CTA per SM, 11 warps with fixed roles:
//   * warps 8 and 10 (loaders): warp 8 fetches units and copies the Q tile
//     and the K tiles of 128 keys, warp 10 the V tiles, all by TMA into
//     128-byte-swizzled shared memory; a K/V tile is gathered through the
//     block table one 16-token block (one box) at a time, blocks past the
//     unit's keys read out of bounds, which fills zeros.  Each unit starts at
//     a different KV tile (rotated by its query tile), so the CTAs that share
//     a kv head do not read the same lines at the same time;
//   * warp 9 (MMA): one thread issues S = Q K^T (both operands in shared
//     memory) and O += P V (P in tensor memory) as tcgen05.mma.kind::f16
//     (bf16 in, fp32 accumulate in tensor memory); S is double-buffered, so
//     S of tile t + 1 is computed while the softmax works on tile t;
//   * warps 0-3 and 4-7: two softmax warpgroups that share every tile:
//     warpgroup w takes its keys 64w .. 64w + 63, thread i owns query row i
//     = TMEM lane i.  The two threads of a row trade their half maxima, so
//     both scale by one running maximum, which moves only when the row's
//     maximum grows by more than 2^8 (base-2 logits): O is rescaled rarely.
//     Each writes its half of P (bf16) over the first half of the tile's S,
//     which both have read by then.  At the end of the unit the two halves'
//     row sums are added and each warpgroup writes half of O's columns.
// An FP8 (E4M3) cache: the loaders copy codes (K to staging buffers, V into
// the V buffers themselves) and the softmax warps widen them to f16, one
// 16-token block per warp, while they work on the tile before; the products
// run as kind::f16.
// Hand-offs are mbarriers; every wait is bounded and a timeout makes the whole
// CTA stop (status PA_DEV_TIMEOUT), drain its copies and MMAs, and free TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kTileM = 128;  // query rows per unit
constexpr int kTileN = 128;  // keys per KV tile
constexpr int kKLoadWarp = 8;   // unit fetch, Q (TMA), K tiles
constexpr int kMmaWarp = 9;
constexpr int kVLoadWarp = 10;  // V tiles
constexpr int kPfThreads = 352;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr float kRescaleThreshold = 8.f;  // base-2 logit growth that forces a rescale

template <int D>
struct PfCfg {
  static constexpr int kRegionBytes = kTileM * 128;     // 128 rows x 64 bf16
  static constexpr int kTileBytes = kTileM * D * 2;     // Q, K or V tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTileBytes;      // K0, K1
  static constexpr int kVOff = kKOff + 2 * kTileBytes;  // V0, V1
  // K and V tiles are stored per 16-token block (one TMA box each):
  //   K [block][8-row group][64-column half][8 rows][128 B]: every 8-key core
  //     group of a column half sits kKGroupBytes after the previous one, as
  //     the K-major operand of S = Q K^T requires;
  //   V [block][64-column half][16 rows][128 B] (MN-major operand of P V).
  static constexpr int kVBlockBytes = kBlockSize * 128 * (D / 64);
  static constexpr int kKGroupBytes = 8 * 128 * (D / 64);
  static constexpr int kSmemBytes = kVOff + 2 * kTileBytes + 1024;  // + alignment slack
  // FP8 cache: a tile's codes are copied by TMA, [16 rows][D bytes] per
  // block, and widened to f16 in the layouts above.  K codes go to two
  // staging buffers ([block][16 rows][D bytes]), so a copy runs two tiles
  // ahead of its widening; V codes go into the upper half of each block's
  // region of the V buffer they are widened into (one warp widens a block in
  // place), so a V copy starts as soon as PV has read that buffer.
  static constexpr int kCodeBytes = kTileN * D;
  static constexpr int kKCodeOff = kVOff + 2 * kTileBytes;
  static constexpr int kSmemBytesF8 = kKCodeOff + 2 * kCodeBytes + 1024;
  // S0, S1 (consecutive tiles) at 0 / 128, each tile's P (bf16 pairs) over the
  // first 64 columns of its S once read; O at 256
  static constexpr int kTmemCols = 512;
  static_assert(D == 64 || D == 128, "head size 64 or 128");
  static_assert(kTileN == kTileM, "K and V tiles share the Q tile geometry");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA exceeds 227 KB");
  // (4 KB: the kernel's static shared memory)
  static_assert(kSmemBytesF8 + 4096 <= 227 * 1024, "shared memory per CTA exceeds 227 KB");
};

// mbarriers.  [2] = one per buffer parity (tile t uses buffers t & 1 of S,
// K, V and P) or per unit slot.  The MMA warp waits once per KV tile t:
// kGo gathers everything O += P V over t and S = Q K^T over t + 2 (same
// buffers) need, so the tensor cores are not left idle between hand-offs.
enum Bar : int {
  kUnitFull = 0,    // [2] unit info published (loader)
  kUnitEmpty = 2,   // [2] unit info read (8 softmax warps, MMA warp, V loader)
  kQFull = 4,       // Q tile landed (TMA)
  kQEmpty = 5,      // every S of the unit done (MMA commit)
  kKFirst = 6,      // [2] the unit's first two K tiles landed (TMA)
  kSFull = 8,       // [2] S = Q K^T done (MMA commit); also frees the K buffer
  kGo = 10,         // [2] tile t: P written and S read (8 softmax warps), V of t landed
                    //     (V loader), K of t + 2 landed or none due (K loader); FP8 cache:
                    //     the softmax warps alone, who also widen K of t + 2 and V of t
  kVLand = 12,      // [2] V tile landed, for a tile whose last block the V loader trims;
                    //     FP8 cache: V codes landed in V buffer 0 / 1
  kPVDone = 14,     // [2] O += P V done (MMA commit); frees the V buffer
  kMx = 16,         // [2] both halves of each row published their maximum (8 warps)
  kMlFull = 18,     // row sums of both halves published (8 warps)
  kMlRead = 19,     // ... and read (8 warps)
  kOFree = 20,      // O read by the epilogue (8 warps)
  kDrain = 21,      // teardown after a timeout
  kPieceDone = 22,  // a split piece's partial state stored (8 softmax warps)
  kPieceLast = 23,  // ... and whether it was the tile's last piece decided (warp 0)
  kQLand = 24,      // FP8 cache: the bf16 Q tile landed (TMA), before its f16 conversion
  kKLand = 25,      // [2] FP8 cache: codes landed in K staging buffer 0 / 1 (TMA)
  kKStFree = 27,    // [2] FP8 cache: K staging buffer 0 / 1 widened by the 8 softmax warps
  kNumBars = 29
};

struct UnitInfo {
  int r, g, a, j0, npos, pos0, kv_end, n_kv;  // r < 0: no more units
  int kt0;                                    // first KV tile (n_kv tiles from there)
  int rot;                                    // KV tile processed first (from kt0)
  int ptile;                                  // query tile index in the step
  int piece, nsplit, slot0;                   // piece of the unit, pieces, slot of piece 0
};

// KV tile processed s-th in unit u (tiles are visited in rotated order).
__device__ __forceinline__ int tile_of(const UnitInfo& u, int s) {
  const int t = s + u.rot;
  return u.kt0 + (t >= u.n_kv ? t - u.n_kv : t);
}

struct PfMaps {
  CUtensorMap q;  // q [T][Hq][D] as 3-D (D, Hq, T), box (64, G, 128/G)
  // bf16 cache:
  CUtensorMap k;  // k_cache as 5-D (64, 8 rows, D/64 halves, 2 row groups, NB x 16 x Hkv),
                  // box (64, 8, D/64, 2, 1) at block x 16 x Hkv + head
  CUtensorMap v;  // v_cache as 5-D (64, 16 rows, D/64 halves, Hkv, NB), box (64, 16, D/64, 1, 1)
  // FP8 cache: k and v as 3-D byte maps (D, 16 rows, NB x 16 x Hkv), box (D, 16, 1) at
  // block x 16 x Hkv + head: one block's codes, [16 rows][D bytes]
};

// max of three floats in one instruction (NaN-free operands here)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// (d0, d1) = (a0, a1) * b + c, one packed instruction for two lanes of work
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n"
      " mov.b64 rc, {%5, %5};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (d0, d1) += (a0, a1)
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1) {
  asm("{\n .reg .b64 ra, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rd, {%0, %1};\n"
      " add.rn.f32x2 rd, rd, ra;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Warp-uniform bounded wait for phase `parity` of `bar`; false after a
// timeout (which it records) or once another role has given up.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort,
                                         int32_t* status) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if (__any_sync(0xffffffffu, *abort != 0)) return false;
  }
  if ((threadIdx.x & 31) == 0) {
    *abort = 1;
    flag_error(status, PA_DEV_TIMEOUT);
  }
  __syncwarp();
  return false;
}

// Arrivals that complete a phase of each barrier.
template <bool F8>
__device__ __forceinline__ uint32_t bar_count(int i) {
  if (i == kUnitEmpty || i == kUnitEmpty + 1) return 10;  // 8 softmax warps, MMA, V loader
  if (i == kGo || i == kGo + 1) return F8 ? 8 : 10;  // 8 softmax warps (+ V and K loaders)
  if (i == kMx || i == kMx + 1 || i == kMlFull || i == kMlRead || i == kOFree ||
      i == kPieceDone || i == kKStFree || i == kKStFree + 1)
    return 8;
  // kQLand, kKLand: TMA (arrive + bytes); kQFull, kKFirst also take the
  // loader's plain arrival after an FP8 conversion: one arrival either way
  return 1;  // TMA (arrive + bytes) or tcgen05.commit
}

// Teardown wait (warp-uniform, bounded, ignores the abort flag).  A kGo
// phase that carried a copy may never complete after an abort (other roles
// stop arriving): the shorter limit still outlasts the copy.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity,
                                           uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return;
}
constexpr uint32_t kGoDrainLimit = 1u << 20;

// One arrival per warp, after every lane's preceding work.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t w;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}
// Two E4M3 codes (low byte first) -> two f16 values, exactly.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t codes16) {
  uint32_t r;
  const uint16_t c = static_cast<uint16_t>(codes16);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(c));
  return r;
}

// FP8: widen blocks b .. b + NB - 1 of a tile of codes at src ([16 rows][D
// bytes] per block, blocks src_stride bytes apart) to f16 at dst, in the
// layout the bf16 TMA copy produces (K: [block][8-row group][64-column half][8 rows][128 B]; V:
// [block][64-column half][16 rows][128 B]; 16-byte chunks XOR-swizzled by
// row); one warp.  A lane converts 16-code chunks (two 16-byte f16 chunks);
// at D = 128 the lanes with the second column half take the neighbouring row
// (parity flipped), so each 8 lanes' loads and stores hit 8 distinct 16-byte
// bank groups.  NB = 2 overlaps two blocks' loads.  Every code is loaded
// before any store, so a block's codes may sit inside its own output.
template <int D, int NB>
__device__ __forceinline__ void widen_blocks(uint32_t src, uint32_t src_stride, uint32_t dst,
                                             bool is_v, int b, int lane) {
  using C = PfCfg<D>;
  constexpr int kRowChunks = D / 16;                 // 16-code chunks per row: 8 or 4
  constexpr int kRowsPerStep = 32 / kRowChunks;      // rows a warp covers per step: 4 or 8
  constexpr int kSteps = kBlockSize / kRowsPerStep;  // steps per block: 4 or 2
  const int c = lane % kRowChunks;
  const int rr = (lane / kRowChunks) ^ (D == 128 ? (c >> 2) & 1 : 0);
  const int half = (c * 16) >> 6;
  uint32_t soff[kSteps][2];  // store offsets within a block
#pragma unroll
  for (int j = 0; j < kSteps; ++j) {
    const int t = j * kRowsPerStep + rr;
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      const int ch = (2 * c + o) & 7;
      const uint32_t sw = static_cast<uint32_t>((ch ^ (t & 7)) << 4);
      soff[j][o] = is_v ? half * (kBlockSize * 128) + t * 128 + sw
                        : (t >> 3) * C::kKGroupBytes + half * 1024 + (t & 7) * 128 + sw;
    }
  }
  const uint32_t lsrc = src + rr * D + c * 16;
  uint4 cv[NB][kSteps];
#pragma unroll
  for (int bb = 0; bb < NB; ++bb)
#pragma unroll
    for (int j = 0; j < kSteps; ++j)
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                   : "=r"(cv[bb][j].x), "=r"(cv[bb][j].y), "=r"(cv[bb][j].z), "=r"(cv[bb][j].w)
                   : "r"(lsrc + (b + bb) * src_stride + j * kRowsPerStep * D)
                   : "memory");
  __syncwarp();
#pragma unroll
  for (int bb = 0; bb < NB; ++bb)
#pragma unroll
    for (int j = 0; j < kSteps; ++j) {
      const uint32_t wd[4] = {cv[bb][j].x, cv[bb][j].y, cv[bb][j].z, cv[bb][j].w};
      uint32_t h[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[2 * e] = e4m3x2_f16x2(wd[e] & 0xffffu);
        h[2 * e + 1] = e4m3x2_f16x2(wd[e] >> 16);
      }
      const uint32_t base = dst + (b + bb) * C::kVBlockBytes;
#pragma unroll
      for (int o = 0; o < 2; ++o)
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(base + soff[j][o]),
                     "r"(h[4 * o]), "r"(h[4 * o + 1]), "r"(h[4 * o + 2]), "r"(h[4 * o + 3])
                     : "memory");
    }
}

}  // namespace

// F8: the cache holds E4M3 codes.  K codes are copied by TMA into two
// staging buffers, two tiles ahead, V codes into the V tile buffers they are
// widened in; both are widened to f16 (exactly) in the K / V tile buffers, a
// unit's first two K tiles by the K loader and every other tile by the
// softmax warps, one block each.  Q is converted from bf16 to f16 in place
// once per unit, and the two products run as kind::f16 with f16 operands (P
// in f16).  The K scale is folded into the softmax scale and the V scale
// into the normalisation.
template <int D, int G, bool F8>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_tc_kernel(const AttnParams p, const __grid_constant__ PfMaps maps) {
  using C = PfCfg<D>;
  constexpr int PM = kTileM / G;  // positions per unit
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ UnitInfo s_units[2];
  __shared__ uint32_t s_tmem;
  __shared__ float s_mx[2][2][kTileM];  // [buffer][column half][row]: half-row maxima
  __shared__ float s_ml[2][kTileM];     // [column half][row]: row sums at the unit's end
  __shared__ int s_abort;
  __shared__ int s_last;  // this CTA's split piece was its query tile's last

  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  volatile int* abort = &s_abort;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), bar_count<F8>(i));
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // Physical block of KV block `lane` (< 8) of tile t, -1 past the unit's
  // keys; checked where it is used, so the load's latency stays hidden.
  auto tile_phys = [&](const UnitInfo& u, int t) {
    const int lb = t * (kTileN / kBlockSize) + lane;
    if (lane < kTileN / kBlockSize && lb * kBlockSize < u.kv_end)
      return __ldg(p.block_tables + static_cast<long long>(u.r) * p.max_blocks_per_seq + lb);
    return -1;
  };
  // TMA copy of KV tile t of unit u into the swizzled buffer at dst: lane
  // b < 8 copies block b, one box (all D columns) per block, in the layouts
  // given with PfCfg; a block past the unit's keys or with a bad table entry
  // is read at index num_blocks (out of bounds: zeros).
  auto copy_kv_tile = [&](const UnitInfo& u, int t, int ph, bool is_v, uint32_t dst,
                          uint32_t full) {
    if (lane < kTileN / kBlockSize && ph != -1 && (ph < 0 || ph >= p.num_blocks)) {
      flag_error(p.status, PA_DEV_BLOCK_RANGE);
      ph = -1;
    }
    if constexpr (F8) {
      // the codes, [16 rows][D bytes] per block: K into the staging buffer
      // at dst, V into the upper half of each block's region of the V
      // buffer at dst
      if (lane == 0) mbar_arrive_expect_tx(full, C::kCodeBytes);
      __syncwarp();
      if (lane < kTileN / kBlockSize) {
        const int coord = ph < 0 ? p.num_blocks : ph;
        const uint32_t d = is_v ? dst + lane * C::kVBlockBytes + C::kVBlockBytes / 2
                                : dst + lane * kBlockSize * D;
        tma_load_3d(d, is_v ? &maps.v : &maps.k, 0, 0,
                    coord * kBlockSize * p.num_kv_heads + u.g, full);
      }
      return;
    }
    if (lane == 0) mbar_arrive_expect_tx(full, C::kTileBytes);
    __syncwarp();
    if (lane < kTileN / kBlockSize) {
      const int coord = ph < 0 ? p.num_blocks : ph;
      if (is_v)
        tma_load_5d(dst + lane * C::kVBlockBytes, &maps.v, 0, 0, 0, u.g, coord, full);
      else
        tma_load_5d(dst + lane * C::kVBlockBytes, &maps.k, 0, 0, 0, 0,
                    coord * kBlockSize * p.num_kv_heads + u.g, full);
    }
  };
  // Rows r0 .. r1 - 1 of the V tile buffer at vb to zeros (all D columns).
  auto zero_v_rows = [&](uint32_t vb, int r0, int r1) {
    constexpr int per_row = (D / 64) * 8;  // 16-byte chunks per row
    for (int idx = lane; idx < (r1 - r0) * per_row; idx += 32) {
      const int row = r0 + idx / per_row, c = idx % per_row;
      asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};\n" ::"r"(
                       vb + (row >> 4) * C::kVBlockBytes + (c >> 3) * (kBlockSize * 128) +
                       (row & 15) * 128 + (c & 7) * 16),
                   "r"(0u)
                   : "memory");
    }
  };
  // FP8: widen a tile of codes at src (blocks src_stride bytes apart) to f16
  // at dst (one warp)
  auto widen_tile = [&](uint32_t src, uint32_t src_stride, uint32_t dst, bool is_v) {
#pragma unroll 1
    for (int b = 0; b < kTileN / kBlockSize; b += 2)
      widen_blocks<D, 2>(src, src_stride, dst, is_v, b, lane);
  };
  // FP8: the landed bf16 Q tile to f16, in place (an element keeps its slot)
  auto q_to_f16 = [&]() {
#pragma unroll 4
    for (int i = lane; i < C::kTileBytes / 16; i += 32) {
      const uint32_t addr = sbase + C::kQOff + i * 16;
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(addr)
                   : "memory");
      const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
      uint32_t h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        h[e] = pack_f16(__uint_as_float(wd[e] << 16), __uint_as_float(wd[e] & 0xffff0000u));
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(h[0]), "r"(h[1]),
                   "r"(h[2]), "r"(h[3])
                   : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
  };

  if (warp == kKLoadWarp) {
    // ------------------------------------------------------------ units, Q, K
    // Work comes in chunks of pieces (PfItem), fetched from a counter: chunk
    // c is pieces starts[c] .. starts[c + 1] - 1 when the plan cut the unit
    // line into chunks, else piece c alone.  (Running a chunk's last piece
    // first, so that a cut unit's two pieces both finish early, measured
    // slower: 200.7 vs 192.5 us on a 2048-token chunk.)
    const int n_chunks = __ldg(p.n_items + (kHdrPrefillChunks - kHdrPrefillItems));
    const bool chunked = __ldg(p.n_items + (kHdrPrefillChunked - kHdrPrefillItems)) != 0;
    const PfItem* pieces = reinterpret_cast<const PfItem*>(p.items);
    const PfTile* qtiles = reinterpret_cast<const PfTile*>(p.tiles);
    int ra = 0, rn = 0, rk = 0;  // the chunk's first piece, its pieces, pieces taken
    // per buffer parity w: nf: first-K copies; sw: S phases waited; ga: kGo
    // arrivals (one per tile of that parity), gk: the last one that carried
    // a copy, plus one
    uint32_t nf[2] = {0, 0}, sw[2] = {0, 0}, ga[2] = {0, 0}, gk[2] = {0, 0}, nq = 0;
    // FP8: code copies issued (copy i: staging buffer i & 1, phase i >> 1); per
    // staging buffer, softmax widenings so far (kStFree phases) and whether
    // its current codes are one of them, not yet waited for
    uint32_t kc = 0, ks0 = 0, ks1 = 0;
    bool kp0 = false, kp1 = false;
    bool q_wait = false;  // FP8: the Q copy not yet waited for
    // The next unit is claimed and published while the current one's last
    // tiles run (before its trailing kGo arrivals), so its metadata loads,
    // Q copy and first K copies are not a serial gap between units; a CTA's
    // first claim is its own index (no atomic), later ones count on from the
    // grid size.  (The mixed step's two 512-token chunks, 256 units of 1-16
    // KV tiles: 30.4 -> 28.8 us.)
    bool first_claim = true;
    auto claim = [&](int ucn, UnitInfo& u) -> bool {
      int pc = -1;
      while (true) {
        if (rk < rn) {
          pc = ra + rk++;
          break;
        }
        int c = 0;
        if (first_claim) {
          c = blockIdx.x;
          first_claim = false;
        } else {
          if (lane == 0) c = static_cast<int>(gridDim.x) + atomicAdd(p.next, 1);
          c = __shfl_sync(0xffffffffu, c, 0);
        }
        if (c >= n_chunks) break;
        ra = chunked ? __ldg(p.order + c) : c;
        rn = (chunked ? __ldg(p.order + c + 1) : c + 1) - ra;
        rk = 0;
      }
      u.r = -1;
      if (pc >= 0) {
        const int4 ta = __ldg(&pieces[pc].a), tb = __ldg(&pieces[pc].b);
        const int4 qt = __ldg(reinterpret_cast<const int4*>(qtiles + ta.x));  // PfTile
        const int S = __ldg(p.seq_lens + qt.x);
        const int a = __ldg(p.qsl + qt.x);
        const int L = __ldg(p.qsl + qt.x + 1) - a;
        u.r = qt.x;
        u.g = ta.y;
        u.a = a;
        u.j0 = qt.y * PM;
        u.npos = min(PM, L - u.j0);
        u.pos0 = S - L + u.j0;
        u.kt0 = ta.z;
        u.n_kv = ta.w - ta.z;
        u.kv_end = min(u.pos0 + u.npos, ta.w * kTileN);  // this piece's keys end here
        u.rot = qt.y % u.n_kv;
        u.ptile = ta.x;
        u.piece = tb.x;
        u.nsplit = tb.y;
        u.slot0 = tb.z;
      }
      const int slot = ucn & 1;
      if (ucn >= 2 && !wait_bar(bar(kUnitEmpty + slot), ((ucn >> 1) - 1) & 1, abort, p.status))
        return false;
      if (lane == 0) {
        s_units[slot] = u;
        mbar_arrive(bar(kUnitFull + slot));
      }
      return true;
    };
    UnitInfo u;
    if (claim(0, u)) for (int uc = 0;; ++uc) {
      if (u.r < 0) break;
      int ph = tile_phys(u, tile_of(u, 0));
      // FP8: K codes of tile sq (tiles in order) into staging buffer kc & 1,
      // once the softmax warps have widened what it held, if theirs.  The
      // loader widens a unit's first two tiles itself (they start the unit);
      // the softmax warps widen tile sq >= 2 while they work on tile sq - 2.
      const uint32_t c0 = kc;
      auto copy_codes = [&](int sq) -> bool {
        const uint32_t b = kc & 1;
        if ((b ? kp1 : kp0) &&
            !wait_bar(bar(kKStFree + b), ((b ? ks1 : ks0) - 1) & 1, abort, p.status))
          return false;
        copy_kv_tile(u, tile_of(u, sq), ph, false, sbase + C::kKCodeOff + b * C::kCodeBytes,
                     bar(kKLand + b));
        const bool soft = sq >= 2;
        if (b) {
          kp1 = soft;
          ks1 += soft;
        } else {
          kp0 = soft;
          ks0 += soft;
        }
        ++kc;
        if (sq + 1 < u.n_kv) ph = tile_phys(u, tile_of(u, sq + 1));
        return true;
      };
      bool ok = true;
      if constexpr (F8) ok = copy_codes(0) && (u.n_kv < 2 || copy_codes(1));  // ahead of Q
      if (!ok) break;
      // Q tile: rows (position, head) of 128/G tokens x G heads, one box per 64 columns
      if (uc > 0 && !wait_bar(bar(kQEmpty), (uc - 1) & 1, abort, p.status)) break;
      const uint32_t q_bar = F8 ? bar(kQLand) : bar(kQFull);
      if (lane == 0) {
        mbar_arrive_expect_tx(q_bar, C::kTileBytes);
#pragma unroll
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sbase + C::kQOff + h * C::kRegionBytes, &maps.q, h * 64, u.g * G,
                      u.a + u.j0, q_bar);
      }
      ++nq;
      q_wait = F8;
      if constexpr (F8) {  // Q to f16 while the codes are on their way
        if (!wait_bar(bar(kQLand), (nq - 1) & 1, abort, p.status)) {
          ok = false;
        } else {
          q_wait = false;
          q_to_f16();
          if (lane == 0) mbar_arrive(bar(kQFull));
        }
      }
      if constexpr (F8) {
        // the first two tiles into K buffers 0 / 1 (freed by the previous
        // unit: its last S of each parity was waited below), then every
        // later tile's codes as their staging buffer frees up
        for (int sq = 0; ok && sq < min(2, u.n_kv); ++sq) {
          const uint32_t i = c0 + sq;
          ++nf[sq];
          if (!wait_bar(bar(kKLand + (i & 1)), (i >> 1) & 1, abort, p.status)) { ok = false; break; }
          widen_tile(sbase + C::kKCodeOff + (i & 1) * C::kCodeBytes, kBlockSize * D,
                     sbase + C::kKOff + sq * C::kTileBytes, false);
          fence_proxy_async_smem();  // the generic-proxy writes, before the tensor cores read them
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kKFirst + sq));
          if (sq + 2 < u.n_kv && !copy_codes(sq + 2)) ok = false;  // into the buffer just read
        }
        for (int sq = 4; ok && sq < u.n_kv; ++sq)
          if (!copy_codes(sq)) ok = false;
        for (int t = 0; t < u.n_kv - 2; ++t) ++sw[t & 1];  // S phases not waited for
      } else {
        // K of tile sq goes into buffer w = sq & 1.  The first two were freed
        // by the previous unit (its last S of each parity was waited below);
        // later ones wait for S of tile sq - 2 and then count as that tile's
        // kGo arrival (bytes included)
        for (int sq = 0; ok && sq < u.n_kv; ++sq) {
          const int w = sq & 1;
          uint32_t full = bar(kKFirst + w);
          if (sq >= 2) {
            if (!wait_bar(bar(kSFull + w), sw[w] & 1, abort, p.status)) { ok = false; break; }
            ++sw[w];
            full = bar(kGo + w);
            gk[w] = ++ga[w];
          } else {
            ++nf[w];
          }
          copy_kv_tile(u, tile_of(u, sq), ph, false, sbase + C::kKOff + w * C::kTileBytes, full);
          if (sq + 1 < u.n_kv) ph = tile_phys(u, tile_of(u, sq + 1));
        }
      }
      UnitInfo nu;
      if (ok) ok = claim(uc + 1, nu);
      // the unit's last two S done (K buffers free for the next unit); bf16:
      // tiles with no K two places on make a plain kGo arrival then
      for (int t = max(0, u.n_kv - 2); ok && t < u.n_kv; ++t) {
        const int w = t & 1;
        if (!wait_bar(bar(kSFull + w), sw[w] & 1, abort, p.status)) { ok = false; break; }
        ++sw[w];
        if constexpr (!F8) {
          ++ga[w];
          warp_arrive(bar(kGo + w));
        }
      }
      if (!ok) break;
      u = nu;
    }
    if (*abort) {  // let every copy issued land before the CTA ends
      if constexpr (F8) {
        if (q_wait) drain_wait(bar(kQLand), (nq - 1) & 1);
        // the last copy into each staging buffer (one at most is in flight per buffer)
        for (uint32_t i = kc > 2 ? kc - 2 : 0; i < kc; ++i)
          drain_wait(bar(kKLand + (i & 1)), (i >> 1) & 1);
      } else {
        if (nq > 0) drain_wait(bar(kQFull), (nq - 1) & 1);
        for (int w = 0; w < 2; ++w) {
          if (nf[w] > 0) drain_wait(bar(kKFirst + w), (nf[w] - 1) & 1);
          if (gk[w] > 0) drain_wait(bar(kGo + w), (gk[w] - 1) & 1, kGoDrainLimit);
        }
      }
    }
    __syncwarp();
  } else if (warp == kVLoadWarp) {
    // ------------------------------------------------------------ V
    // per buffer parity: nv: V tiles (= kGo arrivals); gv: the last kGo phase
    // that carried a copy, plus one; nl: kVLand copies
    uint32_t nv[2] = {0, 0}, gv[2] = {0, 0}, nl[2] = {0, 0};
    bool landing = false;  // a kVLand copy not yet waited for
    int land_w = 0;
    bool vland = false;  // FP8: a code copy into V buffer vland_w not yet drained
    int vland_w = 0;
    for (int uc = 0;; ++uc) {
      const int slot = uc & 1;
      if (!wait_bar(bar(kUnitFull + slot), (uc >> 1) & 1, abort, p.status)) break;
      const UnitInfo u = s_units[slot];
      warp_arrive(bar(kUnitEmpty + slot));
      if (u.r < 0) break;
      int ph = tile_phys(u, tile_of(u, 0));
      bool ok = true;
      if constexpr (F8) {
        // each tile's codes into V buffer w = sq & 1 once PV of the previous
        // tile of that parity is done; the softmax warps widen them there
        for (int sq = 0; sq < u.n_kv; ++sq) {
          const int w = sq & 1;
          if (nv[w] > 0 && !wait_bar(bar(kPVDone + w), (nv[w] - 1) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          copy_kv_tile(u, tile_of(u, sq), ph, true, sbase + C::kVOff + w * C::kTileBytes,
                       bar(kVLand + w));
          ++nv[w];
          vland = true;
          vland_w = w;
          if (sq + 1 < u.n_kv) ph = tile_phys(u, tile_of(u, sq + 1));
        }
      } else {
        for (int sq = 0; sq < u.n_kv; ++sq) {
          const int w = sq & 1;
          const int kt = tile_of(u, sq);
          // V buffer w is free once PV of the previous tile of that parity is done
          if (nv[w] > 0 && !wait_bar(bar(kPVDone + w), (nv[w] - 1) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          const uint32_t vb = sbase + C::kVOff + w * C::kTileBytes;
          if (kt != u.kt0 + u.n_kv - 1 || (u.kv_end & (kBlockSize - 1)) == 0) {
            copy_kv_tile(u, kt, ph, true, vb, bar(kGo + w));  // this tile's kGo arrival
            gv[w] = nv[w] + 1;
          } else {
            // the unit's last block is partial: its rows past the last key
            // (unwritten slots) are zeroed once the tile has landed, so that
            // p = 0 never meets a NaN there; then the kGo arrival
            copy_kv_tile(u, kt, ph, true, vb, bar(kVLand + w));
            landing = true;
            land_w = w;
            if (!wait_bar(bar(kVLand + w), nl[w] & 1, abort, p.status)) { ok = false; break; }
            landing = false;
            ++nl[w];
            const int r0 = u.kv_end - kt * kTileN;
            zero_v_rows(vb, r0, (r0 + kBlockSize - 1) & ~(kBlockSize - 1));
            fence_proxy_async_smem();
            warp_arrive(bar(kGo + w));
          }
          ++nv[w];
          if (sq + 1 < u.n_kv) ph = tile_phys(u, tile_of(u, sq + 1));
        }
      }
      if (!ok) break;
    }
    if (*abort) {
      if (landing) drain_wait(bar(kVLand + land_w), nl[land_w] & 1);
      // FP8: the last code copy into each V buffer
      if (vland) {
        drain_wait(bar(kVLand + vland_w), (nv[vland_w] - 1) & 1);
        if (nv[vland_w ^ 1] > 0) drain_wait(bar(kVLand + (vland_w ^ 1)), (nv[vland_w ^ 1] - 1) & 1);
      }
      for (int w = 0; w < 2; ++w)
        if (gv[w] > 0) drain_wait(bar(kGo + w), (gv[w] - 1) & 1, kGoDrainLimit);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // Kept lean: every cycle this warp spends between products is tensor-core
    // idle time (the issue queue is shallow).  Counters live in registers,
    // descriptors are built once and advanced by their address field.
    constexpr uint32_t kIdS = idesc_kind_f16(kTileM, kTileN, 0, F8);
    constexpr uint32_t kIdPV = idesc_kind_f16(kTileM, D, 1, F8);
    const uint64_t dq = smem_desc_sw128(sbase + C::kQOff, 16, 1024);
    const uint64_t dk = smem_desc_sw128(sbase + C::kKOff, 16, C::kKGroupBytes);
    const uint64_t dv = smem_desc_sw128(sbase + C::kVOff, kBlockSize * 128, 1024);
    // byte offset -> descriptor start-address field (16-byte units; no carry:
    // shared addresses stay below 2^18)
    auto adv = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
    // S = Q K^T of tile t into S buffer w (K buffer w)
    auto mma_s = [&](int w) {
      const uint64_t kb = adv(dk, w * C::kTileBytes);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        // 16 columns: column half kk / 4 (a Q region, or 1 KB into a K group)
        const uint32_t c32 = (kk & 3) * 32;
        tc_mma_f16(tmem + w * kTileN, adv(dq, (kk >> 2) * C::kRegionBytes + c32),
                   adv(kb, (kk >> 2) * 1024 + c32), kIdS, kk > 0);
      }
      tc_commit(bar(kSFull + w));
    };
    // O += P V of a tile: P (bf16 pairs, 8 columns per 16 keys) in the first
    // 64 columns of S buffer w, V in buffer w; first: O is overwritten
    auto mma_pv = [&](int w, bool first) {
      const uint64_t vb = adv(dv, w * C::kTileBytes);
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        tc_mma_f16_ts(tmem + 256, tmem + w * kTileN + kk * 8, adv(vb, kk * C::kVBlockBytes), kIdPV,
                      (first && kk == 0) ? 0u : 1u);
      tc_commit(bar(kPVDone + w));
    };
    uint32_t g0 = 0, g1 = 0;    // tiles per buffer parity so far (kGo phases)
    uint32_t nf0 = 0, nf1 = 0;  // first-K copies per buffer parity so far
    bool ok = true;
    for (int uc = 0; ok; ++uc) {
      const int slot = uc & 1;
      if (!wait_bar(bar(kUnitFull + slot), (uc >> 1) & 1, abort, p.status)) break;
      const UnitInfo u = s_units[slot];
      warp_arrive(bar(kUnitEmpty + slot));
      if (u.r < 0) break;
      const int nkv = u.n_kv;
      if (!wait_bar(bar(kQFull), uc & 1, abort, p.status)) break;
      // The unit's first two S wait for their K copies (S of the previous
      // unit was read before that unit's last kGo); later S(t + 2) go right
      // behind PV(t), both covered by kGo of t.
      if (!wait_bar(bar(kKFirst), nf0 & 1, abort, p.status)) break;
      ++nf0;
      tc_fence_after();
      if (lane == 0) mma_s(0);
      __syncwarp();
      if (nkv > 1) {
        if (!wait_bar(bar(kKFirst + 1), nf1 & 1, abort, p.status)) break;
        ++nf1;
        tc_fence_after();
        if (lane == 0) mma_s(1);
        __syncwarp();
      }
      if (nkv <= 2) {
        if (lane == 0) tc_commit(bar(kQEmpty));
        __syncwarp();
      }
      // PV(t) goes before S(t + 2), which overwrites the P that PV(t) reads
      // (the tensor cores run one thread's MMAs in order); S(t + 1) is
      // computed while the softmax works on t
      for (int t = 0; t < nkv; ++t) {
        const int w = t & 1;
        const uint32_t g = w ? g1 : g0;
        if (!wait_bar(bar(kGo + w), g & 1, abort, p.status)) { ok = false; break; }
        // the previous unit's epilogue must have read O before it is overwritten
        if (t == 0 && uc > 0 && !wait_bar(bar(kOFree), (uc - 1) & 1, abort, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          mma_pv(w, t == 0);
          if (t + 2 < nkv) {
            mma_s(w);
            if (t + 2 == nkv - 1) tc_commit(bar(kQEmpty));
          }
        }
        __syncwarp();
        if (w) ++g1; else ++g0;
      }
    }
    if (*abort) {  // every MMA issued must finish before TMEM is released
      if (lane == 0) tc_commit(bar(kDrain));
      __syncwarp();
      drain_wait(bar(kDrain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Warpgroup w takes keys 64w .. 64w + 63 of every tile; thread i owns
    // query row i = TMEM lane i.  The two threads of a row trade their half
    // maxima through shared memory (kMx), so both use one running maximum
    // and their P halves, O and the row sums share one scale.
    const int w = warp >> 2;       // warpgroup = column half
    const int i = tid & 127;       // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tmem_o = tmem + 256 + lane_off;
    constexpr int kOCols = D / 2;  // O columns this group rescales and writes
    const float sl2 = p.scale_log2;
    const int Hq = p.num_q_heads;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    uint32_t nb0 = 0, nb1 = 0;  // tiles per buffer parity so far (all units)
    uint32_t cb = 0;            // FP8: tiles of earlier units (the code copy index of tile 0)
    uint32_t npieces = 0;       // split pieces finished so far
    const int Hkv = p.num_kv_heads;
    // Merge of a split unit, by its last piece: this thread's row i and its
    // warpgroup's half of the columns, from every piece's (max, sum) and
    // unnormalised O (fp32, in L2); piece sp's state is in slot slot0 + sp.
    auto merge_row = [&](const UnitInfo& u, long long tok, int hh) {
      const long long rbase = u.slot0;
      auto ml_of = [&](int sp) {
        return __ldcg(reinterpret_cast<const float2*>(p.part_ml) +
                      ((rbase + sp) * kTileM + i));
      };
      float M = -CUDART_INF_F;
      for (int sp = 0; sp < u.nsplit; ++sp) M = fmaxf(M, ml_of(sp).x);
      float den = 0.f;
      for (int sp = 0; sp < u.nsplit; ++sp) {
        const float2 ml = ml_of(sp);
        den = fmaf(ml.y, ex2(ml.x - M), den);  // 0 for a piece without visible keys
      }
      const float inv = p.out_scale / den;
      __nv_bfloat16* orow = out + (tok * Hq + u.g * G + hh) * D;
#pragma unroll 1
      for (int c0 = w * kOCols; c0 < (w + 1) * kOCols; c0 += 32) {
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
        for (int sp = 0; sp < u.nsplit; ++sp) {
          const float f = ex2(ml_of(sp).x - M);
          const float4* src = reinterpret_cast<const float4*>(
              p.part_acc + ((rbase + sp) * kTileM + i) * D + c0);
          float4 v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + j);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc[4 * j] = fmaf(v[j].x, f, acc[4 * j]);
            acc[4 * j + 1] = fmaf(v[j].y, f, acc[4 * j + 1]);
            acc[4 * j + 2] = fmaf(v[j].z, f, acc[4 * j + 2]);
            acc[4 * j + 3] = fmaf(v[j].w, f, acc[4 * j + 3]);
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_uint4(pack_bf16(acc[8 * j] * inv, acc[8 * j + 1] * inv),
                              pack_bf16(acc[8 * j + 2] * inv, acc[8 * j + 3] * inv),
                              pack_bf16(acc[8 * j + 4] * inv, acc[8 * j + 5] * inv),
                              pack_bf16(acc[8 * j + 6] * inv, acc[8 * j + 7] * inv));
      }
    };
    for (int uc = 0;; ++uc) {
      const int slot = uc & 1;
      if (!wait_bar(bar(kUnitFull + slot), (uc >> 1) & 1, abort, p.status)) break;
      const UnitInfo u = s_units[slot];
      warp_arrive(bar(kUnitEmpty + slot));
      if (u.r < 0) break;
      const int jj = i / G;
      const bool row_ok = jj < u.npos;
      const int my_pos = u.pos0 + jj;
      float m_used = -CUDART_INF_F, l_part = 0.f;
      bool ok = true;
      for (int t = 0; t < u.n_kv; ++t) {  // t: place in the unit's order
        const int b = t & 1;
        const uint32_t nb = b ? nb1 : nb0;  // uses of buffer b so far
        const int kt = tile_of(u, t);
        const int key0 = kt * kTileN + w * 64;  // first key of this half
        const uint32_t tmem_s = tmem + b * kTileN + lane_off;
        if (!wait_bar(bar(kSFull + b), nb & 1, abort, p.status)) { ok = false; break; }
        tc_fence_after();

        // 64 keys of the S row -> registers, masked (causal edge or padding
        // row: keys past lim) and turned into base-2 logits there
        const bool masked = key0 + 63 > u.pos0 || !row_ok;
        const int lim = row_ok ? my_pos - key0 : -1;
        const float mul = masked ? 1.f : sl2;
        uint32_t sr[64];
        PA_TMEM_LD32(tmem_s + w * 64, sr);
        PA_TMEM_LD32(tmem_s + w * 64 + 32, (sr + 32));
        tmem_wait_ld();
        float mx;
        {
          float m4[4];
          if (masked) {
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const float x = c <= lim ? __uint_as_float(sr[c]) * sl2 : -CUDART_INF_F;
              sr[c] = __float_as_uint(x);
              m4[c & 3] = fmaxf(m4[c & 3], x);
            }
            mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = __uint_as_float(sr[e]);
            if (sl2 >= 0.f) {
#pragma unroll
              for (int c = 4; c < 64; c += 2)
                m4[(c >> 1) & 3] = max3(m4[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
              mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
            } else {
#pragma unroll
              for (int c = 4; c < 64; c += 2)
                m4[(c >> 1) & 3] = min3(m4[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
              mx = fminf(fminf(m4[0], m4[1]), fminf(m4[2], m4[3])) * sl2;
            }
          }
        }
        // the row's maximum over the whole tile: trade halves with the partner
        // thread (both have read their S by then, so P may overwrite it after)
        s_mx[b][w][i] = mx;
        warp_arrive(bar(kMx + b));
        if (!wait_bar(bar(kMx + b), nb & 1, abort, p.status)) { ok = false; break; }
        mx = fmaxf(mx, s_mx[b][w ^ 1][i]);
        float f = 1.f;  // this tile's rescale of the row's earlier state
        if (mx > m_used + kRescaleThreshold) {
          f = ex2(m_used - mx);  // 0 while the row had no visible key
          l_part *= f;
          m_used = mx;
        }
        // P = exp2(logit - m) as bf16 pairs into columns 32w .. 32w + 31 of S
        // buffer b (keys 64w .. 64w + 63 of the tile)
        {
          const float m_sub = m_used == -CUDART_INF_F ? 0.f : m_used;
          float ps4[4] = {0.f, 0.f, 0.f, 0.f};  // two packed pair sums
          uint32_t pw[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float x0, x1;
            fma2(x0, x1, __uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]), mul, -m_sub);
            const float p0 = ex2(x0), p1 = ex2(x1);
            add2(ps4[2 * (c & 1)], ps4[2 * (c & 1) + 1], p0, p1);
            pw[c] = F8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
          }
          PA_TMEM_ST32(tmem_s + w * 32, pw);
          l_part += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
        }
        if constexpr (F8) {
          // this warp's 16-token block of K(t + 2), from its staging buffer
          // into K buffer b (S(t), its last reader, is done), and of V(t), in
          // place in V buffer b (PV(t - 2), its last reader, finished before
          // S(t)); V rows past the unit's last key (unwritten slots) become
          // zeros, so p = 0 never meets a NaN there
          if (t + 2 < u.n_kv) {
            const uint32_t ci = cb + t + 2;
            if (!wait_bar(bar(kKLand + (ci & 1)), (ci >> 1) & 1, abort, p.status)) {
              ok = false;
              break;
            }
            widen_blocks<D, 1>(sbase + C::kKCodeOff + (ci & 1) * C::kCodeBytes, kBlockSize * D,
                               sbase + C::kKOff + b * C::kTileBytes, false, warp, lane);
            warp_arrive(bar(kKStFree + (ci & 1)));
          }
          {
            if (!wait_bar(bar(kVLand + b), nb & 1, abort, p.status)) { ok = false; break; }
            const uint32_t vb = sbase + C::kVOff + b * C::kTileBytes;
            widen_blocks<D, 1>(vb + C::kVBlockBytes / 2, C::kVBlockBytes, vb, true, warp, lane);
            const int r0 = u.kv_end - kt * kTileN;
            if (r0 < kTileN && (r0 >> 4) == warp) {
              __syncwarp();
              zero_v_rows(vb, r0, (r0 + kBlockSize - 1) & ~(kBlockSize - 1));
            }
          }
          fence_proxy_async_smem();  // generic-proxy writes, before the tensor cores read them
        }
        // rescale this group's O columns in rows whose maximum moved, once
        // PV(t - 1) is done (not on the unit's first tile: PV(0) overwrites O)
        if (t > 0 && __any_sync(0xffffffffu, f != 1.f)) {
          const int pb = b ^ 1;
          const uint32_t npv = (pb ? nb1 : nb0) - 1;  // PV(t - 1) is that buffer's last use
          if (!wait_bar(bar(kPVDone + pb), npv & 1, abort, p.status)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < kOCols; c0 += 32) {
            uint32_t o[32];
            PA_TMEM_LD32(tmem_o + w * kOCols + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
            PA_TMEM_ST32(tmem_o + w * kOCols + c0, o);
          }
          tmem_wait_st();
        }
        tmem_wait_st();  // P (and O) stores complete
        tc_fence_before();
        warp_arrive(bar(kGo + b));  // S read, P written, O rescaled
        if (b) ++nb1; else ++nb0;
      }
      if (!ok) break;
      cb += u.n_kv;

      // ---- both halves' row sums (traded while the last PV runs), then
      // this group's half of the O columns
      s_ml[w][i] = l_part;
      warp_arrive(bar(kMlFull));
      if (!wait_bar(bar(kMlFull), uc & 1, abort, p.status)) break;
      const float l_sum = l_part + s_ml[w ^ 1][i];
      warp_arrive(bar(kMlRead));
      {
        const int lb = (u.n_kv - 1) & 1;  // buffer of the last tile: its PV covers all
        const uint32_t npv = (lb ? nb1 : nb0) - 1;
        if (!wait_bar(bar(kPVDone + lb), npv & 1, abort, p.status)) break;
      }
      tc_fence_after();
      const float inv = p.out_scale / l_sum;
      const long long tok = u.a + u.j0 + jj;
      __nv_bfloat16* orow = out + (tok * Hq + u.g * G + (i - jj * G)) * D;
      // a piece of a split query tile keeps its state: unnormalised O and
      // the row's (maximum used, sum) go to its partial slot
      const bool split = u.nsplit > 1;
      const long long prow = static_cast<long long>(u.slot0 + u.piece) * kTileM + i;
#pragma unroll
      for (int c0 = w * kOCols; c0 < (w + 1) * kOCols; c0 += 32) {
        uint32_t o[32];
        PA_TMEM_LD32(tmem_o + c0, o);
        tmem_wait_ld();
        if (row_ok && split) {
          float4* dst = reinterpret_cast<float4*>(p.part_acc + prow * D + c0);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                 __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
        } else if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(o[8 * j + e]) * inv;
            dst[j] = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
                                pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
          }
        }
      }
      if (split && row_ok && w == 0)
        reinterpret_cast<float2*>(p.part_ml)[prow] = make_float2(m_used, l_sum);
      tc_fence_before();
      warp_arrive(bar(kOFree));
      // neither group publishes its next unit's row sum before both read these
      if (!wait_bar(bar(kMlRead), uc & 1, abort, p.status)) break;
      if (split) {
        // every piece counts itself in once its state is stored; the last one
        // (of any CTA) merges the tile's pieces
        __threadfence();
        warp_arrive(bar(kPieceDone));
        if (warp == 0) {
          if (!wait_bar(bar(kPieceDone), npieces & 1, abort, p.status)) break;
          if (lane == 0) {
            __threadfence();
            s_last = atomicAdd(p.merge_cnt + u.ptile * Hkv + u.g, 1) == u.nsplit - 1;
            mbar_arrive(bar(kPieceLast));
          }
          __syncwarp();
        }
        if (!wait_bar(bar(kPieceLast), npieces & 1, abort, p.status)) break;
        const bool last = *reinterpret_cast<volatile int*>(&s_last) != 0;
        ++npieces;
        if (last) {
          __threadfence();
          if (row_ok) merge_row(u, tok, i - jj * G);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// bf16 tensor map with 128-byte swizzle and zero fill out of bounds.
bool encode_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  const auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
             const_cast<void*>(base), dims, strides_bytes, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Byte (uint8) tensor map with no swizzle and zero fill out of bounds (FP8 codes).
bool encode_map_u8(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                   const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  const auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank),
             const_cast<void*>(base), dims, strides_bytes, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int D, int G, bool F8>
cudaError_t launch_pf(const AttnParams& p, int num_sms, cudaStream_t stream) {
  using C = PfCfg<D>;
  constexpr int kSmem = F8 ? C::kSmemBytesF8 : C::kSmemBytes;
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<D, G, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  PfMaps maps;
  const cuuint64_t e2 = 2;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(p.num_q_heads),
                                static_cast<cuuint64_t>(p.num_tokens)};
    const cuuint64_t strides[2] = {D * e2, static_cast<cuuint64_t>(p.num_q_heads) * D * e2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kTileM / G)};
    if (!encode_map(&maps.q, p.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  if constexpr (F8) {
    // codes of one (block, head): 16 rows of D bytes at a stride of Hkv x D;
    // the last index steps one head (D bytes), as in the bf16 K map
    const cuuint64_t hkv = static_cast<cuuint64_t>(p.num_kv_heads);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(kBlockSize),
                                static_cast<cuuint64_t>(p.num_blocks) * kBlockSize * hkv};
    if (dims[2] + hkv > 0x7fffffffull) return cudaErrorInvalidValue;
    const cuuint64_t strides[2] = {hkv * D, static_cast<cuuint64_t>(D)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(kBlockSize), 1};
    if (!encode_map_u8(&maps.k, p.k_cache, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_map_u8(&maps.v, p.v_cache, 3, dims, strides, box)) return cudaErrorInvalidValue;
  } else {
    const cuuint64_t hkv = static_cast<cuuint64_t>(p.num_kv_heads);
    const cuuint64_t row = hkv * D * e2;  // bytes between a block's rows
    // K: (64 columns, 8 rows, D/64 halves, 2 row groups, block x 16 x Hkv + head);
    // the last index steps one head (D x 2 bytes), so a block's box for head
    // g starts at block x 16 x Hkv + g and a block index past the pool reads
    // out of bounds.  Coordinates are 32-bit.
    const cuuint64_t kdims[5] = {64, 8, static_cast<cuuint64_t>(D / 64), 2,
                                 static_cast<cuuint64_t>(p.num_blocks) * kBlockSize * hkv};
    if (kdims[4] + hkv > 0x7fffffffull) return cudaErrorInvalidValue;
    const cuuint64_t kstrides[4] = {row, 128, 8 * row, D * e2};
    const cuuint32_t kbox[5] = {64, 8, static_cast<cuuint32_t>(D / 64), 2, 1};
    if (!encode_map(&maps.k, p.k_cache, 5, kdims, kstrides, kbox)) return cudaErrorInvalidValue;
    // V: (64 columns, 16 rows, D/64 halves, kv head, block); the halves
    // dimension's stride (128 B) is below the rows' (Hkv x D x 2 B)
    const cuuint64_t vdims[5] = {64, static_cast<cuuint64_t>(kBlockSize),
                                 static_cast<cuuint64_t>(D / 64), hkv,
                                 static_cast<cuuint64_t>(p.num_blocks)};
    const cuuint64_t vstrides[4] = {hkv * D * e2, 128, D * e2, kBlockSize * hkv * D * e2};
    const cuuint32_t vbox[5] = {64, static_cast<cuuint32_t>(kBlockSize),
                                static_cast<cuuint32_t>(D / 64), 1, 1};
    if (!encode_map(&maps.v, p.v_cache, 5, vdims, vstrides, vbox)) return cudaErrorInvalidValue;
  }
  prefill_tc_kernel<D, G, F8><<<num_sms, kPfThreads, kSmem, stream>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace

namespace {
template <bool F8>
cudaError_t launch_pf_dtype(const AttnParams& p, int head_size, int group, int num_sms,
                            cudaStream_t stream) {
  if (head_size == 128) {
    switch (group) {
      case 1: return launch_pf<128, 1, F8>(p, num_sms, stream);
      case 2: return launch_pf<128, 2, F8>(p, num_sms, stream);
      case 4: return launch_pf<128, 4, F8>(p, num_sms, stream);
      case 8: return launch_pf<128, 8, F8>(p, num_sms, stream);
    }
  } else if (head_size == 64) {
    switch (group) {
      case 1: return launch_pf<64, 1, F8>(p, num_sms, stream);
      case 2: return launch_pf<64, 2, F8>(p, num_sms, stream);
      case 4: return launch_pf<64, 4, F8>(p, num_sms, stream);
      case 8: return launch_pf<64, 8, F8>(p, num_sms, stream);
    }
  }
  return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_prefill_tc(const AttnParams& p, int head_size, int group, int num_sms,
                              bool fp8_cache, cudaStream_t stream) {
  return fp8_cache ? launch_pf_dtype<true>(p, head_size, group, num_sms, stream)
                   : launch_pf_dtype<false>(p, head_size, group, num_sms, stream);
}

}  // namespace pa
