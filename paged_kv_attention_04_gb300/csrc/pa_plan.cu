// Step planning on the device: no host<->device copy is needed to split the
// step's requests into work.
//
// The step is one flattened super-sequence: decodes first, then prefill
// chunks ("Serving models at scale with vLLM", section Chunked prefill;
// "Inside vLLM", section Run forward pass).  One CTA reads seq_lens and
// query_start_loc, checks them, sorts every request into a class
//   decode   q_len == 1
//   small    1 < q_len < prefill_min_qlen (CUDA-core tiles of a few positions)
//   prefill  q_len >= prefill_min_qlen   (tensor-core tiles)
// and writes the work lists the attention kernels consume, plus zeroed
// per-tile split counters.  A decode or small tile whose KV is longer than
// `bps` blocks is split into several items whose partial softmax states are
// merged by the last item to finish.  Decode items are handed out in a
// dispatch order: items of at least half a split first, in request order
// (short items among them would only add their fixed cost late), then the
// shorter ones largest first (a counting sort by blocks), so the last units
// the CTAs pick up are short and the step ends evenly.
//
// Tensor-core prefill units (query tile x kv head) are scheduled one of three
// ways, by what the step holds (each measured best for its kind of step):
//   * fewer units than SMs (a short chunk after a long prompt): each unit's
//     KV is cut into pieces sized for one round, one piece per SM;
//   * long units, a few per SM (a long chunk): McNaughton's wrap-around rule
//     for identical machines with preemption -- the units are laid end to
//     end on a line (each its KV tiles plus a fixed cost), the line is cut
//     into equal chunks, one per SM, and a unit a cut falls inside becomes
//     pieces (a cut that would leave a piece under kMinPrefillSplitTiles KV
//     tiles moves to the unit's edge), so every CTA streams the same number
//     of KV tiles instead of some SMs running one unit more than the rest;
//   * otherwise whole units, handed out last first (within a chunk later
//     query tiles see more keys, and later chunks carry more prior context),
//     whose dynamic fetch already evens out many short units.
// The pieces of a cut unit keep partial softmax states that the last one to
// finish merges.
#include <climits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

// One CTA of 256 threads: a step's requests are walked 256 at a time.  The
// plan's phases are barrier- and latency-bound, so a smaller CTA plans
// faster (measured: the TinyLlama step 35.2 -> 33.2 us, the tiny fp32 step
// 18.8 -> 16.7 us against 1024 threads; larger steps unchanged).
#ifndef PA_PLAN_THREADS
#define PA_PLAN_THREADS 256
#endif
constexpr int kPlanThreads = PA_PLAN_THREADS;
static_assert(kPlanThreads % 32 == 0 && kPlanThreads <= 1024, "whole warps, one CTA");
constexpr int kShortItems = 2048;  // short decode items listed in shared memory (else re-read)

#ifndef PA_UNITS_PER_CTA
#define PA_UNITS_PER_CTA 8  // split-size target: decode units per CTA (see plan_kernel)
#endif
#ifndef PA_SMALL_SPLIT_PCT
#define PA_SMALL_SPLIT_PCT 150  // small-step decode split, % of the even per-CTA share
#endif
#ifndef PA_SPLIT_MIN
#define PA_SPLIT_MIN 16  // smallest decode split (blocks)
#endif

// decode items, decode tiles, small items, small tiles, prefill line length, long decode
// items, prefill query tiles
constexpr int kLists = 7;


// Exclusive scan of kLists ints per thread across the CTA, all lists at once;
// `total` receives each list's CTA total.
__device__ void block_exclusive_scan(int (&v)[kLists], int (*warp_sums)[kLists],
                                     int (&total)[kLists]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x[kLists];
#pragma unroll
  for (int k = 0; k < kLists; ++k) x[k] = v[k];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < kLists; ++k) {
      const int y = __shfl_up_sync(0xffffffffu, x[k], o);
      if (lane >= o) x[k] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int k = 0; k < kLists; ++k) warp_sums[warp][k] = x[k];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < kLists; ++k) {
      int w = (lane < (kPlanThreads / 32)) ? warp_sums[lane][k] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane][k] = w;  // inclusive
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kLists; ++k) {
    v[k] = (warp > 0 ? warp_sums[warp - 1][k] : 0) + x[k] - v[k];
    total[k] = warp_sums[kPlanThreads / 32 - 1][k];
  }
  __syncthreads();
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// KV blocks per split for a request with nb KV blocks: at least bps, large
// enough that a tile has at most kMaxSplits splits, at most kMaxUnitBlocks.
__device__ __forceinline__ int request_bps(int nb, int bps) {
  return min(max(bps, ceil_div(nb, kMaxSplits)), kMaxUnitBlocks);
}

// Number of KV splits of a tile whose last query row sits at position pos_last.
__device__ __forceinline__ int splits_for(int pos_last, int bps) {
  return ceil_div(ceil_div(pos_last + 1, kBlockSize), bps);
}

}  // namespace

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p) {
  __shared__ int warp_sums[32][kLists];
  __shared__ int carry[kLists];
  __shared__ int err;
  __shared__ int size_hist[kMaxUnitBlocks + 1];  // short decode items per size (blocks)
  __shared__ unsigned long long s_blocks;        // KV blocks of the requests that split
  __shared__ unsigned long long s_blocks_d;      // ... of the decode requests among them
  __shared__ int2 s_short[kShortItems];          // short decode items: (item, blocks)
  __shared__ int s_nshort;
  static_assert(kMaxUnitBlocks == 8 * 32, "the dispatch-order scan gives each lane 8 sizes");
  // The attention kernel that follows may become resident now; it waits for
  // this grid to finish before it reads the work lists.  This grid itself may
  // have started early (programmatic launch) beside the previous kernel in
  // the stream, normally the slot write.  It reads only seq_lens and
  // query_start_loc, which that kernel does not write, and writes only the
  // workspace, which no kernel still running reads (the slot write starts only
  // after the previous step's kernels have finished).  So it plans at once and
  // waits for the previous kernel only before finishing: the attention kernel
  // then sees the slot write complete as well.
  launch_dependents();
  const int B = p.num_seqs;
  // This thread's first request (r = threadIdx.x), loaded before the set-up
  // barrier so that the load's latency overlaps it; both passes below reuse
  // it (r < kPlanThreads is that request), later requests are loaded there.
  int pre_s = 0, pre_a = 0, pre_b = 0;
  if (static_cast<int>(threadIdx.x) < B) {
    pre_s = __ldg(p.seq_lens + threadIdx.x);
    pre_a = __ldg(p.qsl + threadIdx.x);
    pre_b = __ldg(p.qsl + threadIdx.x + 1);
  }
  auto load_request = [&](int r, int& S, int& qa, int& qb) {
    if (r < kPlanThreads) {
      S = pre_s;
      qa = pre_a;
      qb = pre_b;
    } else {
      S = __ldg(p.seq_lens + r);
      qa = __ldg(p.qsl + r);
      qb = __ldg(p.qsl + r + 1);
    }
  };
  char* ws = p.ws;
  int* hdr = reinterpret_cast<int*>(ws + p.lay.hdr);
  int4* items_d = reinterpret_cast<int4*>(ws + p.lay.items_d);
  int4* tiles_d = reinterpret_cast<int4*>(ws + p.lay.tiles_d);
  int4* items_s = reinterpret_cast<int4*>(ws + p.lay.items_s);
  int4* tiles_s = reinterpret_cast<int4*>(ws + p.lay.tiles_s);
  UnitRec* recs_d = reinterpret_cast<UnitRec*>(ws + p.lay.recs_d);
  UnitRec* recs_s = reinterpret_cast<UnitRec*>(ws + p.lay.recs_s);
  int* cnt_d = reinterpret_cast<int*>(ws + p.lay.cnt_d);
  int* cnt_s = reinterpret_cast<int*>(ws + p.lay.cnt_s);
  PfTile* tiles_p = reinterpret_cast<PfTile*>(ws + p.lay.tiles_p);
  PfItem* items_p = reinterpret_cast<PfItem*>(ws + p.lay.items_p);
  int* starts_p = reinterpret_cast<int*>(ws + p.lay.starts_p);
  int* cnt_p = reinterpret_cast<int*>(ws + p.lay.cnt_p);
  int* order_d = reinterpret_cast<int*>(ws + p.lay.order_d);

  for (int i = threadIdx.x; i <= kMaxUnitBlocks; i += kPlanThreads) size_hist[i] = 0;
  if (threadIdx.x == 0) {
    err = 0;
    s_blocks = 0;
    s_blocks_d = 0;
    s_nshort = 0;
    for (int i = 0; i < kLists; ++i) carry[i] = 0;
  }
  __syncthreads();

  // Split size for this step: at least p.bps blocks, and longer when the
  // CTAs would otherwise get more than ~8 units each of the decode and
  // few-token KV (measured: longer units amortise each unit's fixed cost once
  // there are enough of them), up to kMaxUnitBlocks.
  // Out-of-range lengths are left out here (they are flagged below).
  {
    unsigned long long mine = 0, mine_d = 0;
    for (int r = threadIdx.x; r < B; r += kPlanThreads) {
      int S, qa, qb;
      load_request(r, S, qa, qb);
      // the ends of query_start_loc, checked by the threads that load them
      if ((r == 0 && qa != 0) || (r == B - 1 && qb != p.num_tokens)) atomicOr(&err, PA_DEV_QSL);
      const int L = qb - qa;
      if (S < 1 || S > p.max_seq_len || L < 1 || L > S) continue;
      if (L < p.prefill_min_qlen) {
        mine += static_cast<unsigned long long>(ceil_div(S, kBlockSize));
        if (L == 1) mine_d += static_cast<unsigned long long>(ceil_div(S, kBlockSize));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mine += __shfl_down_sync(0xffffffffu, mine, o);
      mine_d += __shfl_down_sync(0xffffffffu, mine_d, o);
    }
    if ((threadIdx.x & 31) == 0 && mine) atomicAdd(&s_blocks, mine);
    if ((threadIdx.x & 31) == 0 && mine_d) atomicAdd(&s_blocks_d, mine_d);
  }
  __syncthreads();
  const int num_ctas = max(1, p.num_ctas);
  const long long per_cta = static_cast<long long>(s_blocks) * p.num_kv_heads / num_ctas;
  const int bps = static_cast<int>(
      min(static_cast<long long>(kMaxUnitBlocks),
          max(static_cast<long long>(p.bps), (per_cta + PA_UNITS_PER_CTA - 1) / PA_UNITS_PER_CTA)));
  // Decode splits of a small step (fewer KV blocks x heads than one
  // p.bps-block split per CTA): with whole-request units most CTAs would sit
  // idle while a few stream the longest requests, so the split is sized to
  // give about one unit per CTA (PA_SMALL_SPLIT_PCT % of the even share), at
  // least PA_SPLIT_MIN blocks, and large enough that the items fit the
  // workspace: items <= requests + blocks / split.
  int bps_d = bps;
  {
    const long long total_d = static_cast<long long>(s_blocks_d) * p.num_kv_heads;
    if (total_d < static_cast<long long>(num_ctas) * p.bps) {
      const long long want = (total_d * PA_SMALL_SPLIT_PCT + 100LL * num_ctas - 1) / (100LL * num_ctas);
      const long long room = p.cap.decode_items - B;
      const long long need = room > 0 ? (static_cast<long long>(s_blocks_d) + room - 1) / room
                                       : static_cast<long long>(p.bps);
      bps_d = static_cast<int>(min(static_cast<long long>(p.bps),
                                   max(max(want, need), static_cast<long long>(PA_SPLIT_MIN))));
    }
  }

  // One pass: classify and count, exclusive-scan the counts across the CTA,
  // and let each request's thread write its own items and tiles at its
  // offsets (every write checked against the list's capacity).
  int carry_r[kLists] = {0, 0, 0, 0, 0, 0, 0};
  for (int base = 0; base < B; base += kPlanThreads) {
    const int r = base + threadIdx.x;
    int c = kClassNone;
    int cnt[kLists] = {0, 0, 0, 0, 0, 0, 0};
    int S = 0, a = 0, L = 0;
    if (r < B) {
      int b;
      load_request(r, S, a, b);
      L = b - a;
      int e = 0;
      if (L < 0 || a < 0 || b > p.num_tokens) e |= PA_DEV_QSL;
      else if (L < 1 || L > S || S > p.max_seq_len || L > p.max_query_len ||
               ceil_div(S, kBlockSize) > p.max_blocks_per_seq)
        e |= PA_DEV_LENGTHS;
      if (e) {
        atomicOr(&err, e);
      } else if (L == 1) {
        c = kClassDecode;
        cnt[1] = 1;
        const int nb = ceil_div(S, kBlockSize), rb = request_bps(nb, bps_d);
        cnt[0] = splits_for(S - 1, rb);
        // long items: every full split, and the last one if it is at least half a split
        cnt[5] = cnt[0] - 1 + (2 * (nb - (cnt[0] - 1) * rb) >= bps_d ? 1 : 0);
      } else if (L >= p.prefill_min_qlen) {
        c = kClassPrefill;
        const int pm = p.prefill_rows / p.group;
        cnt[6] = ceil_div(L, pm);
        // line length of the request's units (query tiles x kv heads)
        for (int m = 0; m < cnt[6]; ++m)
          cnt[4] += ceil_div(S - L + min(L, (m + 1) * pm), kPrefillKeys) + kPrefillUnitCost;
        cnt[4] *= p.num_kv_heads;
      } else {
        c = kClassSmall;
        cnt[3] = ceil_div(L, p.small_positions);
        const int rb = request_bps(ceil_div(S, kBlockSize), bps);
        for (int m = 0; m < cnt[3]; ++m) {
          const int last = min(L, (m + 1) * p.small_positions) - 1;
          cnt[2] += splits_for(S - L + last, rb);
        }
      }
    }
    int off[kLists], tot[kLists];
#pragma unroll
    for (int k = 0; k < kLists; ++k) off[k] = cnt[k];
    block_exclusive_scan(off, warp_sums, tot);
#pragma unroll
    for (int k = 0; k < kLists; ++k) off[k] += carry_r[k];
    if (c == kClassDecode) {
      // items off[0] .. off[0] + cnt[0] - 1: one split of the request each
      const int tile = off[1];
      const int nb = ceil_div(S, kBlockSize);
      const int rb = request_bps(nb, bps_d);
      const int ns = cnt[0];
      if (tile < p.cap.decode_tiles) tiles_d[tile] = make_int4(off[0], ns, rb, 0);
      for (int s = 0; s < ns; ++s) {
        const int i = off[0] + s;
        if (i >= p.cap.decode_items) break;
        items_d[i] = make_int4(r, 0, s * rb, tile);
        const int b0 = s * rb, b1 = min(b0 + rb, nb);
        // long items take dispatch slots in request order (they are a prefix
        // of the request's splits, and off[5] + s <= i); short ones are counted
        if (s < cnt[5]) order_d[off[5] + s] = i;
        else {
          atomicAdd(&size_hist[b1 - b0], 1);
          const int j = atomicAdd(&s_nshort, 1);
          if (j < kShortItems) s_short[j] = make_int2(i, b1 - b0);
        }
        recs_d[i].a = make_int4(r, 0, b0, b1);
        recs_d[i].b = make_int4(tile, off[0], ns, a);
        recs_d[i].c = make_int4(1, S - 1, min(b1 * kBlockSize, S), 0);
      }
    } else if (c == kClassSmall) {
      // tiles of small_positions positions, each expanded into its splits
      const int rb = request_bps(ceil_div(S, kBlockSize), bps);
      const int P = p.small_positions;
      int first = off[2];
      for (int m = 0; m < cnt[3]; ++m) {
        const int tile = off[3] + m;
        const int ns = splits_for(S - L + min(L, (m + 1) * P) - 1, rb);
        const int npos = min(P, L - m * P);
        const int pos0 = S - L + m * P;
        const int kv_end = pos0 + npos;
        const int nblk = ceil_div(kv_end, kBlockSize);
        if (tile < p.cap.small_tiles) tiles_s[tile] = make_int4(first, ns, rb, 0);
        for (int s = 0; s < ns && first + s < p.cap.small_items; ++s) {
          items_s[first + s] = make_int4(r, m, s * rb, tile);
          const int b0 = s * rb, b1 = min(b0 + rb, nblk);
          recs_s[first + s].a = make_int4(r, m * P, b0, b1);
          recs_s[first + s].b = make_int4(tile, first, ns, a);
          recs_s[first + s].c = make_int4(npos, pos0, min(b1 * kBlockSize, kv_end), 0);
        }
        first += ns;
      }
    } else if (c == kClassPrefill) {
      // tensor-core query tiles of prefill_rows rows (positions x grouped
      // heads), laid on the line from the request's offset
      const int pm = p.prefill_rows / p.group;
      int x = off[4];
      for (int m = 0; m < cnt[6]; ++m) {
        const int q = off[6] + m;
        const int nkv = ceil_div(S - L + min(L, (m + 1) * pm), kPrefillKeys);
        if (q < p.cap.prefill_tiles) tiles_p[q] = PfTile{r, m, nkv, x};
        x += (nkv + kPrefillUnitCost) * p.num_kv_heads;
      }
    }
#pragma unroll
    for (int k = 0; k < kLists; ++k) carry_r[k] += tot[k];
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < kLists; ++k) carry[k] = carry_r[k];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (carry[0] > p.cap.decode_items || carry[1] > p.cap.decode_tiles ||
        carry[2] > p.cap.small_items || carry[3] > p.cap.small_tiles ||
        carry[6] > p.cap.prefill_tiles)
      err |= PA_DEV_CAPACITY;
  }
  __syncthreads();
  if (err & (PA_DEV_CAPACITY | PA_DEV_QSL)) {
    // Nothing is safe to schedule: publish empty lists.
    if (threadIdx.x == 0) {
      for (int i = 0; i < kHdrWords; ++i) hdr[i] = 0;
      flag_error(p.status, err);
    }
    wait_prior_grid();
    return;
  }
  const int n_di = carry[0], n_dt = carry[1], n_si = carry[2], n_st = carry[3];
  const int n_pt = carry[6];

  // Prefill pieces (see the file comment), one thread per unit u = q x Hkv + g.
  const int Hkv = p.num_kv_heads;
  const int line = carry[4];
  const int n_units = n_pt * Hkv;
  const int kv_tiles = line / Hkv - kPrefillUnitCost * n_pt;  // KV tiles of all query tiles
  const int P = max(1, p.num_sms);
  bool chunked = false;
  int tps = INT_MAX, n_ch = 0, clen = 1;
  if (n_units > 0 && n_units < P) {
    // one round: pieces x heads <= units + KV tiles x heads / tps <= SMs, and
    // the pieces with a partial state (<= that sum) within the slots
    const long long kvh = static_cast<long long>(kv_tiles) * Hkv;
    const long long room = p.cap.prefill_slots - n_units;
    if (room > 0) {
      const long long want = (kvh + (P - n_units) - 1) / (P - n_units);
      const long long need = (kvh + room - 1) / room;
      tps = static_cast<int>(min(static_cast<long long>(INT_MAX),
                                 max(max(want, need), static_cast<long long>(kMinPrefillSplitTiles))));
    }
    // tps bounds the pieces from the mean; the longest piece decides the
    // round, so take the smallest size that still fits: thread i tries
    // tps - i, counting its pieces (and partial slots) over the query tiles
    // (64 tokens after 32768 and 16 after 98304: pieces of at most 70 KV
    // tiles instead of 77, 120.4 -> 119.0 us)
    __shared__ int s_nkv[kPlanThreads];
    __shared__ int s_tps;
    if (tps != INT_MAX && n_pt <= kPlanThreads) {
      if (threadIdx.x < n_pt) s_nkv[threadIdx.x] = max(1, tiles_p[threadIdx.x].nkv);
      if (threadIdx.x == 0) s_tps = tps;
      __syncthreads();
      const int T = tps - static_cast<int>(threadIdx.x);
      if (T >= kMinPrefillSplitTiles) {
        long long pieces = 0, slots = 0;
        for (int q = 0; q < n_pt; ++q) {
          const int k = ceil_div(s_nkv[q], T);
          pieces += k;
          slots += k > 1 ? k : 0;
        }
        if (pieces * Hkv <= P && slots * Hkv <= p.cap.prefill_slots) atomicMin(&s_tps, T);
      }
      __syncthreads();
      tps = s_tps;
    }
  } else if (n_units >= P && n_units <= kPrefillChunkMaxWaves * P &&
             kv_tiles >= kPrefillChunkMinTiles * n_pt && p.cap.prefill_slots >= 2) {
    // chunks of clen line positions, clen >= the unit cost + two minimum
    // pieces, so the cut-or-snap rule keeps chunk starts in order; fewer than
    // half the slots, since the pieces of cut units number at most 2 x cuts
    chunked = true;
    const int want = static_cast<int>(min(static_cast<long long>(min(kPrefillMaxChunks, P)),
                                          p.cap.prefill_slots / 2));
    clen = max(ceil_div(line, want), kPrefillUnitCost + 2 * kMinPrefillSplitTiles);
    n_ch = ceil_div(line, clen);
  }
  int n_rec = 0, n_slot = 0;
  for (int base = 0; base < n_units; base += kPlanThreads) {
    const int u = base + threadIdx.x;
    int v[kLists] = {0, 0, 0, 0, 0, 0, 0}, tot[kLists];
    PfTile t{0, 0, 0, 0};
    int g = 0, s0 = 0, e0 = 0, c0 = 0, nrec = 0;
    if (u < n_units) {
      t = tiles_p[u / Hkv];  // written above by this CTA
      g = u % Hkv;
      s0 = t.x + g * (t.nkv + kPrefillUnitCost);
      e0 = s0 + t.nkv + kPrefillUnitCost;
      if (chunked) {
        // cuts: the chunk starts c x clen in [s0 + cost + min piece, e0 - min piece]
        c0 = ceil_div(s0 + kPrefillUnitCost + kMinPrefillSplitTiles, clen);
        nrec = max(0, (e0 - kMinPrefillSplitTiles) / clen - c0 + 1) + 1;
      } else {
        nrec = t.nkv > tps ? ceil_div(t.nkv, tps) : 1;
      }
      v[0] = nrec;
      v[1] = nrec > 1 ? nrec : 0;
    }
    block_exclusive_scan(v, warp_sums, tot);
    if (u < n_units) {
      const int rec0 = n_rec + v[0];
      const int slot0 = nrec > 1 ? n_slot + v[1] : -1;
      const int per = ceil_div(t.nkv, nrec);
      for (int k = 0; k < nrec; ++k) {
        int kt0, kt1;
        if (chunked) {
          kt0 = k == 0 ? 0 : (c0 + k - 1) * clen - s0 - kPrefillUnitCost;
          kt1 = k == nrec - 1 ? t.nkv : (c0 + k) * clen - s0 - kPrefillUnitCost;
        } else {
          kt0 = k * per;
          kt1 = min(t.nkv, (k + 1) * per);
        }
        // whole units are handed out last first
        const int idx = (!chunked && tps == INT_MAX) ? n_units - 1 - u : rec0 + k;
        if (idx < p.cap.prefill_pieces) {
          PfItem it;
          it.a = make_int4(u / Hkv, g, kt0, kt1);
          it.b = make_int4(k, nrec, slot0, 0);
          items_p[idx] = it;
        }
      }
      if (chunked) {
        // the chunk starts falling in this unit: cut, or moved to an edge
        for (int c = max(1, ceil_div(s0, clen)); c < n_ch && c * clen < e0; ++c) {
          const int b = c * clen;
          starts_p[c] = b - s0 < kPrefillUnitCost + kMinPrefillSplitTiles ? rec0
                        : e0 - b < kMinPrefillSplitTiles                 ? rec0 + nrec
                                                                         : rec0 + c - c0 + 1;
        }
      }
    }
    n_rec += tot[0];
    n_slot += tot[1];
  }
  if (threadIdx.x == 0) {
    if (chunked) {
      starts_p[0] = 0;
      starts_p[n_ch] = n_rec;
    } else {
      n_ch = n_rec;
    }
    if (n_rec > p.cap.prefill_pieces || n_slot > p.cap.prefill_slots) err |= PA_DEV_CAPACITY;
  }
  __syncthreads();
  if (err & PA_DEV_CAPACITY) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < kHdrWords; ++i) hdr[i] = 0;
      flag_error(p.status, err);
    }
    wait_prior_grid();
    return;
  }
  // dispatch order (it does not change results: partial states are stored
  // and merged by item, in split order).  The long items took the first
  // n_long slots above; short items: exclusive scan of the size histogram
  // from the largest size down (each bucket's first slot), then every short
  // item takes the next slot of its bucket
  const int n_long = carry[5];
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) tot += size_hist[kMaxUnitBlocks - (8 * lane + j)];
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = n_long + incl - tot;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int sz = kMaxUnitBlocks - (8 * lane + j);
      const int c = size_hist[sz];
      size_hist[sz] = run;
      run += c;
    }
  }
  __syncthreads();
  if (s_nshort <= kShortItems) {
    for (int j = threadIdx.x; j < s_nshort; j += kPlanThreads) {
      const int2 e = s_short[j];
      order_d[atomicAdd(&size_hist[e.y], 1)] = e.x;
    }
  } else {
    for (int i = threadIdx.x; i < n_di; i += kPlanThreads) {
      // short = under half a split (full splits hold at least bps_d blocks)
      const int4 a = recs_d[i].a;  // written above by this CTA
      if (2 * (a.w - a.z) < bps_d) order_d[atomicAdd(&size_hist[a.w - a.z], 1)] = i;
    }
  }
  for (int i = threadIdx.x; i < n_dt * p.num_kv_heads; i += kPlanThreads) cnt_d[i] = 0;
  for (int i = threadIdx.x; i < n_st * p.num_kv_heads; i += kPlanThreads) cnt_s[i] = 0;
  for (int i = threadIdx.x; i < n_pt * p.num_kv_heads; i += kPlanThreads) cnt_p[i] = 0;
  if (threadIdx.x == 0) {
    hdr[kHdrDecodeItems] = n_di;
    hdr[kHdrDecodeTiles] = n_dt;
    hdr[kHdrDecodeNext] = 0;
    hdr[kHdrSmallItems] = n_si;
    hdr[kHdrSmallTiles] = n_st;
    hdr[kHdrSmallNext] = 0;
    hdr[kHdrPrefillItems] = n_pt;
    hdr[kHdrPrefillNext] = 0;
    hdr[kHdrPrefillChunks] = n_ch;
    hdr[kHdrPrefillChunked] = chunked ? 1 : 0;
    if (err) flag_error(p.status, err);
  }
  wait_prior_grid();
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, p);
}

}  // namespace pa
