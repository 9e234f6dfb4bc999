// Host side of the libpa C ABI: argument checks, workspace layout, launch
// order.  Nothing here touches tensor data; every step of the attention runs
// in the kernels.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "pa_internal.h"

namespace pa {
cudaError_t launch_attn_mma_bf16(const AttnParams& p, int head_size, int group, int positions,
                                 bool keys_as_m, int num_sms, cudaStream_t stream,
                                 int* grid_only);
cudaError_t launch_attn_cc_f32(const AttnParams& p, int head_size, int group, int positions,
                               int num_sms, cudaStream_t stream, int* grid_only);

cudaError_t launch_attn_by_dtype(const AttnParams& p, pa_dtype dtype, int head_size, int group,
                                 int positions, bool keys_as_m, int num_sms, cudaStream_t stream,
                                 int* grid_only) {
  return dtype == PA_BF16 ? launch_attn_mma_bf16(p, head_size, group, positions, keys_as_m,
                                                 num_sms, stream, grid_only)
                          : launch_attn_cc_f32(p, head_size, group, positions, num_sms, stream,
                                               grid_only);
}

namespace {

thread_local std::string g_last_error;
thread_local cudaEvent_t g_prof_start = nullptr;
thread_local cudaEvent_t g_prof_stop = nullptr;
thread_local cudaEvent_t g_pf_prof_start = nullptr;
thread_local cudaEvent_t g_pf_prof_stop = nullptr;
thread_local bool g_prefill_overlap = true;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int elem_bytes(pa_dtype t) { return t == PA_FP8_E4M3 ? 1 : (t == PA_BF16 ? 2 : 4); }

bool fp8_cache(const pa_layout* L) { return L->cache_dtype == PA_FP8_E4M3; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

int check_layout(const pa_layout* L) {
  if (!L) return fail(PA_ERR_INVALID, "layout is NULL");
  if (L->dtype != PA_F32 && L->dtype != PA_BF16)
    return fail(PA_ERR_INVALID, "dtype %d is not PA_F32 or PA_BF16", static_cast<int>(L->dtype));
  if (L->cache_dtype != L->dtype) {
    if (L->cache_dtype != PA_FP8_E4M3)
      return fail(PA_ERR_INVALID, "cache_dtype %d must equal dtype or be PA_FP8_E4M3",
                  static_cast<int>(L->cache_dtype));
    if (L->dtype != PA_BF16)
      return fail(PA_ERR_UNSUPPORTED, "an FP8 cache is built for bf16 q/k/v only");
    if (!(std::isfinite(L->k_scale) && L->k_scale > 0.f && std::isfinite(L->v_scale) &&
          L->v_scale > 0.f))
      return fail(PA_ERR_INVALID, "FP8 cache scales must be finite and positive");
  }
  if (L->num_q_heads <= 0 || L->num_kv_heads <= 0 || L->head_size <= 0 || L->num_blocks <= 0)
    return fail(PA_ERR_INVALID, "heads, head_size and num_blocks must be positive");
  if (L->num_q_heads % L->num_kv_heads)
    return fail(PA_ERR_INVALID, "num_q_heads %d is not a multiple of num_kv_heads %d",
                L->num_q_heads, L->num_kv_heads);
  if (L->block_size != kBlockSize)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (built for 16)", L->block_size);
  if (L->head_size != 64 && L->head_size != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_size %d (built for 64 and 128)", L->head_size);
  const int g = L->num_q_heads / L->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return fail(PA_ERR_UNSUPPORTED, "GQA group %d (built for 1, 2, 4, 8)", g);
  if (static_cast<long long>(L->num_blocks) * kBlockSize > (1LL << 40))
    return fail(PA_ERR_INVALID, "num_blocks %d too large", L->num_blocks);
  return PA_OK;
}

#ifndef PA_SPLIT_BLOCKS
#define PA_SPLIT_BLOCKS 128
#endif

// Smallest KV split, in blocks (the plan grows it for steps with much KV per
// CTA).  A decode unit's cost is set by its blocks (instructions and latency
// per block), not its bytes: 128 blocks measured best for bf16 at head size
// 128 and 64 and for FP8 alike.
int blocks_per_split(const pa_layout* L) {
  (void)L;
  int b = PA_SPLIT_BLOCKS;
  if (b > kMaxUnitBlocks) b = kMaxUnitBlocks;
  return b < 1 ? 1 : b;
}

int small_positions(const pa_layout* L) { return kSmallRows / (L->num_q_heads / L->num_kv_heads); }

Capacity capacity(const pa_layout* L, int B, int T, int max_seq_len) {
  Capacity c{};
  const long long max_nb = cdiv(max_seq_len, kBlockSize);
  // most splits any tile gets (see the plan kernel's per-request split size)
  long long splits = cdiv(max_nb, blocks_per_split(L));
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (cdiv(max_nb, kMaxUnitBlocks) > splits) splits = cdiv(max_nb, kMaxUnitBlocks);
  const long long multi = T > B ? (T - B < B ? T - B : B) : 0;  // requests with q_len >= 2
  c.decode_tiles = B;
  // plus room for the finer splits of small steps: the plan keeps a small
  // step's decode items within requests + blocks / split, and raises its
  // split size until they fit this capacity
  c.decode_items = static_cast<long long>(B) * splits + cdiv(kSmallStepUnits, L->num_kv_heads);
  c.small_tiles = (T > B ? cdiv(T - B, small_positions(L)) : 0) + multi;
  c.small_items = c.small_tiles * splits;
  const long long group = L->num_q_heads / L->num_kv_heads;
  c.prefill_tiles = L->dtype == PA_BF16
                        ? cdiv(static_cast<long long>(T) * group, kPrefillRows) + multi : 0;
  // a step that can hold a chunk of kPrefillMinQlen tokens may cut prefill
  // units: at chunk boundaries (a unit with k cuts has k + 1 <= 2k pieces, and
  // a step has fewer chunks than kPrefillMaxChunks and than its longest
  // possible unit line over the shortest chunk, unit cost + two min pieces),
  // or, when units are scarce, into pieces the plan keeps within these slots
  c.prefill_pieces = c.prefill_tiles * L->num_kv_heads;
  if (c.prefill_tiles > 0 && T - B >= kPrefillMinQlen - 1) {
    const long long line = c.prefill_tiles * L->num_kv_heads *
                           (cdiv(max_seq_len, kPrefillKeys) + kPrefillUnitCost);
    long long chunks = cdiv(line, kPrefillUnitCost + 2 * kMinPrefillSplitTiles);
    if (chunks > kPrefillMaxChunks) chunks = kPrefillMaxChunks;
    c.prefill_slots = 2 * chunks;
    c.prefill_pieces += c.prefill_slots;
  }
  return c;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Per host thread and device: a side stream and two events used to run the
// tensor-core prefill kernel beside the decode kernel (fork after the plan,
// join before returning).  Created on the first call that needs them.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideStream g_side[64];

int side_stream_of_current_device(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(PA_ERR_CUDA, "device ordinal %d", dev);
  SideStream& s = g_side[dev];
  if (!s.stream) {
    e = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail_cuda(e, "side stream set-up");
  }
  *out = &s;
  return PA_OK;
}

int num_sms_of_current_device(int* out) {
  static int cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(PA_ERR_CUDA, "device ordinal %d", dev);
  if (!cache[dev]) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
    cache[dev] = n;
  }
  *out = cache[dev];
  return PA_OK;
}

}  // namespace

int set_last_error(int code, const char* msg) {
  g_last_error = msg;
  return code;
}

WsLayout ws_layout(const Capacity& cap, int Hkv, int D, int group) {
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  const size_t rows_d = static_cast<size_t>(group);
  const size_t rows_s = static_cast<size_t>(kSmallRows);
  w.hdr = take(kHdrWords * sizeof(int));
  w.items_d = take(sizeof(int4) * cap.decode_items);
  w.tiles_d = take(sizeof(int4) * cap.decode_tiles);
  w.items_s = take(sizeof(int4) * cap.small_items);
  w.tiles_s = take(sizeof(int4) * cap.small_tiles);
  w.tiles_p = take(sizeof(PfTile) * cap.prefill_tiles);
  w.items_p = take(sizeof(PfItem) * cap.prefill_pieces);
  w.starts_p = take(cap.prefill_tiles > 0 ? sizeof(int) * (kPrefillMaxChunks + 1) : 0);
  w.cnt_p = take(sizeof(int) * cap.prefill_tiles * Hkv);
  w.recs_d = take(sizeof(UnitRec) * cap.decode_items);
  w.recs_s = take(sizeof(UnitRec) * cap.small_items);
  w.order_d = take(sizeof(int) * cap.decode_items);
  w.cnt_d = take(sizeof(int) * cap.decode_tiles * Hkv);
  w.cnt_s = take(sizeof(int) * cap.small_tiles * Hkv);
  w.part_acc_d = take(sizeof(float) * cap.decode_items * Hkv * rows_d * D);
  w.part_ml_d = take(sizeof(float) * cap.decode_items * Hkv * rows_d * 2);
  w.part_acc_s = take(sizeof(float) * cap.small_items * Hkv * rows_s * D);
  w.part_ml_s = take(sizeof(float) * cap.small_items * Hkv * rows_s * 2);
  w.part_acc_p = take(sizeof(float) * cap.prefill_slots * kPrefillRows * D);
  w.part_ml_p = take(sizeof(float) * cap.prefill_slots * kPrefillRows * 2);
  w.total = off;
  return w;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_last_error(void) { return g_last_error.c_str(); }

int pa_version(void) { return 200; }

int pa_set_profile_events(void* start, void* stop) {
  g_prof_start = static_cast<cudaEvent_t>(start);
  g_prof_stop = static_cast<cudaEvent_t>(stop);
  return PA_OK;
}

int pa_set_prefill_profile_events(void* start, void* stop) {
  g_pf_prof_start = static_cast<cudaEvent_t>(start);
  g_pf_prof_stop = static_cast<cudaEvent_t>(stop);
  return PA_OK;
}

int pa_set_prefill_overlap(int on) {
  g_prefill_overlap = on != 0;
  return PA_OK;
}

int pa_cache_write(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                   void* k_cache, void* v_cache, const pa_layout* layout, int32_t* status,
                   void* stream) {
  g_last_error.clear();
  if (int rc = check_layout(layout)) return rc;
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "num_tokens %d < 0", num_tokens);
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PA_ERR_INVALID, "null tensor pointer");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PA_ERR_INVALID, "k, v, k_cache and v_cache must be 16-byte aligned");
  if (!aligned(slot_mapping, 8)) return fail(PA_ERR_INVALID, "slot_mapping must be 8-byte aligned");
  if (status && !aligned(status, 4)) return fail(PA_ERR_INVALID, "status must be 4-byte aligned");
  const int row_bytes = layout->num_kv_heads * layout->head_size * elem_bytes(layout->dtype);
  const long long num_slots = static_cast<long long>(layout->num_blocks) * kBlockSize;
  if (fp8_cache(layout) && !aligned(k_cache, 8)) return fail(PA_ERR_INVALID, "cache alignment");
  cudaError_t e = fp8_cache(layout)
                      ? launch_cache_write_fp8(k, v, slot_mapping, num_tokens, k_cache, v_cache,
                                               row_bytes, num_slots, layout->k_scale,
                                               layout->v_scale, status,
                                               static_cast<cudaStream_t>(stream))
                      : launch_cache_write(k, v, slot_mapping, num_tokens, k_cache, v_cache,
                                           row_bytes, num_slots, status,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cache write launch");
  return PA_OK;
}

size_t pa_forward_workspace_size(const pa_layout* layout, int num_seqs, int num_tokens,
                                 int max_seq_len) {
  g_last_error.clear();
  if (check_layout(layout)) return 0;
  if (num_seqs < 0 || num_tokens < 0 || max_seq_len < 0) {
    fail(PA_ERR_INVALID, "negative size");
    return 0;
  }
  const Capacity cap = capacity(layout, num_seqs, num_tokens, max_seq_len);
  return ws_layout(cap, layout->num_kv_heads, layout->head_size,
                   layout->num_q_heads / layout->num_kv_heads)
      .total;
}

int pa_forward(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
               const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_query_len,
               int max_seq_len, float scale, void* out, void* workspace, size_t workspace_bytes,
               const pa_layout* layout, int32_t* status, void* stream) {
  g_last_error.clear();
  if (int rc = check_layout(layout)) return rc;
  if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || max_seq_len < 0 ||
      max_blocks_per_seq < 0)
    return fail(PA_ERR_INVALID, "negative size argument");
  if (num_seqs == 0 || num_tokens == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start_loc || !out ||
      !workspace)
    return fail(PA_ERR_INVALID, "null pointer argument");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PA_ERR_INVALID, "q, out, k_cache and v_cache must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4))
    return fail(PA_ERR_INVALID, "int32 arrays must be 4-byte aligned");
  if (!aligned(workspace, 256)) return fail(PA_ERR_INVALID, "workspace must be 256-byte aligned");
  if (status && !aligned(status, 4)) return fail(PA_ERR_INVALID, "status must be 4-byte aligned");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "scale is not finite");
  if (max_query_len < 1 || max_seq_len < 1)
    return fail(PA_ERR_INVALID, "max_query_len and max_seq_len must be >= 1");
  if (cdiv(max_seq_len, kBlockSize) > max_blocks_per_seq)
    return fail(PA_ERR_INVALID, "max_blocks_per_seq %d < ceil(max_seq_len / 16) = %lld",
                max_blocks_per_seq, cdiv(max_seq_len, kBlockSize));
  if (num_tokens < num_seqs)
    return fail(PA_ERR_INVALID, "num_tokens %d < num_seqs %d: every request needs a new token",
                num_tokens, num_seqs);
  const int group = layout->num_q_heads / layout->num_kv_heads;
  const Capacity cap = capacity(layout, num_seqs, num_tokens, max_seq_len);
  if (cap.decode_items > (1LL << 30) || cap.small_items > (1LL << 30))
    return fail(PA_ERR_INVALID, "step too large for one call");
  const WsLayout lay = ws_layout(cap, layout->num_kv_heads, layout->head_size, group);
  if (workspace_bytes < lay.total)
    return fail(PA_ERR_INVALID, "workspace of %zu bytes < %zu needed", workspace_bytes, lay.total);
  int num_sms = 0;
  if (int rc = num_sms_of_current_device(&num_sms)) return rc;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  char* ws = static_cast<char*>(workspace);
  int* hdr = reinterpret_cast<int*>(ws + lay.hdr);

  PlanParams pp{};
  pp.seq_lens = seq_lens;
  pp.qsl = query_start_loc;
  pp.num_seqs = num_seqs;
  pp.num_tokens = num_tokens;
  pp.max_query_len = max_query_len;
  pp.max_seq_len = max_seq_len;
  pp.max_blocks_per_seq = max_blocks_per_seq;
  pp.bps = blocks_per_split(layout);
  pp.num_sms = num_sms;
  const bool tc_prefill = layout->dtype == PA_BF16;  // bf16 or FP8 cache
  const bool run_prefill = tc_prefill && max_query_len >= kPrefillMinQlen;
  // bf16 decode tiles: keys as the MMA's M dimension when the step also runs
  // the tensor-core prefill kernel (the decode kernel then shares the GPU and
  // is not purely HBM-bound: the mixed step's decode 258 -> 229 us), query
  // rows as M otherwise (alone, HBM-bound: 225 vs 231 us on Llama-3-8B)
  const bool keys_as_m = run_prefill;
  {
    AttnParams none{};
    e = fp8_cache(layout)
            ? launch_attn_fp8(none, layout->head_size, group, 1, num_sms, st, &pp.num_ctas)
            : launch_attn_by_dtype(none, layout->dtype, layout->head_size, group, 1, keys_as_m,
                                   num_sms, st, &pp.num_ctas);
    if (e != cudaSuccess) return fail_cuda(e, "decode grid size");
  }
  pp.small_positions = small_positions(layout);
  pp.prefill_min_qlen = tc_prefill ? kPrefillMinQlen : 0x7fffffff;
  pp.prefill_rows = kPrefillRows;
  pp.group = group;
  pp.num_kv_heads = layout->num_kv_heads;
  pp.cap = cap;
  pp.ws = ws;
  pp.lay = lay;
  pp.status = status;
  e = launch_plan(pp, st);
  if (e != cudaSuccess) return fail_cuda(e, "plan launch");

  // Chunked prefill (tensor cores) runs on a side stream, launched before the
  // decode kernel so that decode CTAs fill the SMs the prefill CTAs leave:
  // the HBM-bound and the tensor-bound work overlap.  With the overlap off it
  // runs on `st` before the decode kernel.
  const bool fork = run_prefill && g_prefill_overlap;
  SideStream* side = nullptr;
  if (fork) {
    if (int rc = side_stream_of_current_device(&side)) return rc;
  }

  AttnParams ap{};
  ap.q = q;
  ap.k_cache = k_cache;
  ap.v_cache = v_cache;
  ap.block_tables = block_tables;
  ap.seq_lens = seq_lens;
  ap.qsl = query_start_loc;
  ap.out = out;
  ap.max_blocks_per_seq = max_blocks_per_seq;
  ap.num_q_heads = layout->num_q_heads;
  ap.num_kv_heads = layout->num_kv_heads;
  ap.num_blocks = layout->num_blocks;
  ap.num_tokens = num_tokens;
  ap.scale_log2 = scale * 1.4426950408889634f * (fp8_cache(layout) ? layout->k_scale : 1.f);
  ap.out_scale = fp8_cache(layout) ? layout->v_scale : 1.f;
  ap.status = status;

  if (run_prefill) {
    AttnParams pf = ap;
    pf.n_items = hdr + kHdrPrefillItems;
    pf.next = hdr + kHdrPrefillNext;
    pf.items = reinterpret_cast<const int4*>(ws + lay.items_p);  // PfItem pairs
    pf.recs = nullptr;
    pf.tiles = reinterpret_cast<const int4*>(ws + lay.tiles_p);  // PfTile
    pf.order = reinterpret_cast<const int*>(ws + lay.starts_p);  // chunk starts
    pf.merge_cnt = reinterpret_cast<int*>(ws + lay.cnt_p);
    pf.part_acc = reinterpret_cast<float*>(ws + lay.part_acc_p);
    pf.part_ml = reinterpret_cast<float*>(ws + lay.part_ml_p);
    cudaStream_t pst = st;
    if (fork) {
      e = cudaEventRecord(side->fork, st);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
      if (e != cudaSuccess) return fail_cuda(e, "side stream fork");
      pst = side->stream;
    }
    if (g_pf_prof_start) cudaEventRecord(g_pf_prof_start, pst);
    e = launch_prefill_tc(pf, layout->head_size, group, num_sms, fp8_cache(layout), pst);
    if (e != cudaSuccess) return fail_cuda(e, "prefill attention launch");
    if (g_pf_prof_stop) cudaEventRecord(g_pf_prof_stop, pst);
    if (fork) {
      e = cudaEventRecord(side->join, side->stream);
      if (e != cudaSuccess) return fail_cuda(e, "side stream join");
    }
  }

  // decode rows (q_len == 1); the launch may overlap the plan's tail
  ap.after_plan = 1;
  ap.n_items = hdr + kHdrDecodeItems;
  ap.next = hdr + kHdrDecodeNext;
  ap.items = reinterpret_cast<const int4*>(ws + lay.items_d);
  ap.recs = reinterpret_cast<const UnitRec*>(ws + lay.recs_d);
  ap.order = reinterpret_cast<const int*>(ws + lay.order_d);
  ap.tiles = reinterpret_cast<const int4*>(ws + lay.tiles_d);
  ap.merge_cnt = reinterpret_cast<int*>(ws + lay.cnt_d);
  ap.part_acc = reinterpret_cast<float*>(ws + lay.part_acc_d);
  ap.part_ml = reinterpret_cast<float*>(ws + lay.part_ml_d);
  if (g_prof_start) cudaEventRecord(g_prof_start, st);
  e = fp8_cache(layout)
          ? launch_attn_fp8(ap, layout->head_size, group, 1, num_sms, st)
          : launch_attn_by_dtype(ap, layout->dtype, layout->head_size, group, 1, keys_as_m, num_sms,
                                 st);
  if (e != cudaSuccess) return fail_cuda(e, "decode attention launch");
  if (g_prof_stop) cudaEventRecord(g_prof_stop, st);

  if (max_query_len > 1) {
    ap.after_plan = 0;
    ap.n_items = hdr + kHdrSmallItems;
    ap.next = hdr + kHdrSmallNext;
    ap.items = reinterpret_cast<const int4*>(ws + lay.items_s);
    ap.recs = reinterpret_cast<const UnitRec*>(ws + lay.recs_s);
    ap.order = nullptr;
    ap.tiles = reinterpret_cast<const int4*>(ws + lay.tiles_s);
    ap.merge_cnt = reinterpret_cast<int*>(ws + lay.cnt_s);
    ap.part_acc = reinterpret_cast<float*>(ws + lay.part_acc_s);
    ap.part_ml = reinterpret_cast<float*>(ws + lay.part_ml_s);
    e = fp8_cache(layout)
            ? launch_attn_fp8(ap, layout->head_size, group, small_positions(layout), num_sms, st)
            : launch_attn_by_dtype(ap, layout->dtype, layout->head_size, group,
                                   small_positions(layout), false, num_sms, st);
    if (e != cudaSuccess) return fail_cuda(e, "small-q attention launch");
  }
  if (fork) {
    e = cudaStreamWaitEvent(st, side->join, 0);
    if (e != cudaSuccess) return fail_cuda(e, "side stream join wait");
  }
  return PA_OK;
}

}  // extern "C"
