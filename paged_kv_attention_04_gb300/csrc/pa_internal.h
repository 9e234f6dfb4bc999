// Internal declarations shared by the host API and the kernels of libpa.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

constexpr int kBlockSize = 16;        // tokens per KV block
constexpr int kSmallRows = 16;        // query rows (positions x grouped heads) per few-token tile
constexpr int kMaxSplits = 64;        // KV splits per tile are kept at or below this ...
constexpr int kMaxUnitBlocks = 256;   // ... unless a split would exceed this many blocks
constexpr int kPrefillRows = 128;     // query rows per tensor-core prefill tile
constexpr int kPrefillMinQlen = 16;   // bf16 chunks at least this long use the tensor-core kernel
constexpr int kSmallStepUnits = 2048; // extra decode units (items x kv heads) a workspace holds
                                      // for the finer splits of small steps
constexpr int kPrefillKeys = 128;     // keys per KV tile of the tensor-core prefill kernel
// Tensor-core prefill scheduling (see the plan kernel).  A unit is (query tile,
// kv head); its KV tiles may be cut into pieces, each at least
// kMinPrefillSplitTiles tiles, whose partial softmax states the last piece
// merges.  Steps with long units and a few of them per SM are cut by a line
// of units into at most kPrefillMaxChunks equal chunks, a unit taking its KV
// tiles plus kPrefillUnitCost (its fixed cost: Q load, first copies,
// epilogue) on the line.
constexpr int kMinPrefillSplitTiles = 4;
constexpr int kPrefillUnitCost = 4;
constexpr int kPrefillMaxChunks = 320;
constexpr int kPrefillChunkMinTiles = 24;  // chunked when units average at least this many tiles
constexpr int kPrefillChunkMaxWaves = 6;   // ... and number at most this many per SM

// Work-list classes written by the plan kernel.
enum ReqClass : int { kClassNone = 0, kClassDecode = 1, kClassSmall = 2, kClassPrefill = 3 };

// Header words at the start of the workspace.
enum Hdr : int {
  kHdrDecodeItems = 0, kHdrDecodeTiles, kHdrDecodeNext,
  kHdrSmallItems, kHdrSmallTiles, kHdrSmallNext,
  kHdrPrefillItems, kHdrPrefillNext,       // prefill query tiles; chunk counter
  kHdrPrefillChunks, kHdrPrefillChunked,   // chunks; 1: chunk starts listed, 0: a piece each
  kHdrWords = 16
};

// Capacities (host upper bounds) for one step.
struct Capacity {
  long long decode_items, decode_tiles;
  long long small_items, small_tiles;
  long long prefill_tiles;   // query tiles of 128 rows
  long long prefill_pieces;  // units or pieces of their KV
  long long prefill_slots;   // pieces with a partial state (of units cut in several)
};

// Byte offsets of every workspace region (all 256-byte aligned).
struct WsLayout {
  size_t hdr;
  size_t items_d, tiles_d, items_s, tiles_s;
  size_t tiles_p, items_p, starts_p;  // prefill query tiles, pieces, chunk starts
  size_t cnt_p, part_acc_p, part_ml_p;  // prefill merge counters, partial states
  size_t recs_d, recs_s;  // per item: 3 x int4 unit records (see UnitRec)
  size_t order_d;         // decode items in dispatch order (largest split first)
  size_t cnt_d, cnt_s;
  size_t part_acc_d, part_ml_d, part_acc_s, part_ml_s;
  size_t total;
};

struct PlanParams {
  const int32_t* seq_lens;
  const int32_t* qsl;
  int num_seqs, num_tokens, max_query_len, max_seq_len, max_blocks_per_seq;
  int bps;              // KV blocks per split (minimum; long requests use larger splits)
  int num_sms;          // SMs of the device
  int num_ctas;         // CTAs of the decode kernel's grid (the plan sizes splits from the
                        // step's KV per CTA)
  int small_positions;  // query positions per small-q tile
  int prefill_min_qlen; // requests with q_len >= this go to the tensor-core kernel
  int prefill_rows;     // query rows (positions x group) per prefill tile
  int group;            // num_q_heads / num_kv_heads
  int num_kv_heads;
  Capacity cap;
  char* ws;
  WsLayout lay;
  int32_t* status;
};

// Everything a kernel needs to start on one item, precomputed by the plan
// kernel so a work fetch is one load (plus the block-table slice):
//   a = {r, j0 (first query position of the tile), b0, b1 (KV blocks [b0, b1))}
//   b = {tile, first item of the tile, splits of the tile, qsl[r]}
//   c = {valid positions in the tile, position of its first row, one past the
//        last visible key of this split, 0}
struct UnitRec {
  int4 a, b, c;
};

// A tensor-core prefill query tile of the step, in request order then query
// tile m: {r, m, KV tiles its rows see (nkv), line position of its kv-head-0
// unit}.  Its unit for kv head g spans line positions [x + g * len,
// x + (g + 1) * len), len = nkv + kPrefillUnitCost.
struct PfTile {
  int r, m, nkv, x;
};

// One piece of tensor-core prefill work: a = {query tile q, kv head g, first
// KV tile, one past the last KV tile}; b = {piece index, pieces of the unit,
// partial-state slot of piece 0 (-1 for a whole unit: it writes the output),
// 0}.  Piece k uses slot b.z + k.
struct PfItem {
  int4 a, b;
};

// One unit of CUDA-core attention work: request r, query tile m, KV split s,
// and the tile's global index (for the split merge).
struct AttnParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  void* out;
  int max_blocks_per_seq;
  int num_q_heads, num_kv_heads, num_blocks, num_tokens;
  float scale_log2;      // softmax scale * log2(e) (times k_scale for an FP8 cache)
  float out_scale;       // applied to the normalised output (v_scale for an FP8 cache)
  const int* n_items;    // device count of work items (x num_kv_heads units)
  int after_plan;        // host side: launch with a programmatic dependency on the plan
  int* next;             // device work counter (zeroed by the plan kernel)
  const int4* items;     // {r, m, first KV block, tile}
  const UnitRec* recs;   // per item, the same fully decoded
  const int* order;      // dispatch order: the k-th item fetched is order[k] (null: k)
  const int4* tiles;     // {first item, number of splits, KV blocks per split, 0}
                         // (prefill: the query tiles, PfTile)
  int* merge_cnt;        // [tiles][num_kv_heads]
  float* part_acc;       // [items][num_kv_heads][rows][D]
  float* part_ml;        // [items][num_kv_heads][rows][2]
  int32_t* status;
};

// Sets the message pa_last_error() returns on this thread; returns code.
int set_last_error(int code, const char* msg);

// Workspace regions for a step with capacity cap (see pa_forward_workspace_size).
WsLayout ws_layout(const Capacity& cap, int num_kv_heads, int head_size, int group);

// Kernel launchers (return cudaError_t of the launch).
cudaError_t launch_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                               int num_tokens, void* k_cache, void* v_cache, int row_bytes,
                               long long num_slots, int32_t* status, cudaStream_t stream);
// Quantising slot write into an FP8 (E4M3) cache; row_bytes is the bf16 input row.
cudaError_t launch_cache_write_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                                   int num_tokens, void* k_cache, void* v_cache, int row_bytes,
                                   long long num_slots, float k_scale, float v_scale,
                                   int32_t* status, cudaStream_t stream);
cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);
// Tensor-core (tcgen05) chunked-prefill attention over the prefill list
// (bf16 q/out; a bf16 or an FP8 (E4M3) cache).
cudaError_t launch_prefill_tc(const AttnParams& p, int head_size, int group, int num_sms,
                              bool fp8_cache, cudaStream_t stream);
// Split-KV attention over the decode or few-token list, by element type:
// bf16 runs the warp-level tensor-core (mma.sync) kernel, fp32 the CUDA-core
// kernel.  positions: 1 (decode list) or the few-token tile height.
// keys_as_m (bf16 decode tiles): the keys are the MMA's M dimension and the
// query rows its N, instead of the query rows padded to 16 as M.  With
// grid_only set nothing is launched: the grid size (CTAs) the launch would
// use is stored there.  Returns cudaErrorInvalidValue for an unbuilt
// combination.
cudaError_t launch_attn_by_dtype(const AttnParams& p, pa_dtype dtype, int head_size, int group,
                                 int positions, bool keys_as_m, int num_sms, cudaStream_t stream,
                                 int* grid_only = nullptr);
// bf16 q/out over an FP8 (E4M3) cache (tensor-core decode and few-token tiles).
cudaError_t launch_attn_fp8(const AttnParams& p, int head_size, int group, int positions,
                            int num_sms, cudaStream_t stream, int* grid_only = nullptr);

}  // namespace pa
