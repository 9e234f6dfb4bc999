/*
 * pa.h -- C ABI of libpa, paged-KV attention for one continuous-batching step
 * on one GB300 (sm_103a).
 *
 * The step has two calls:
 *   pa_cache_write  writes each new token's K and V into its paged slot;
 *   pa_forward      runs attention for every new token over its request's
 *                   KV, read through the request's block table.
 *
 * Sources (page title, section):
 *   "Inside vLLM: Anatomy of a High-Throughput LLM Inference System",
 *     LLM Engine constructor: a KV block is 2 (K/V) x block_size (16) x
 *       num_kv_heads x head_size x dtype bytes;
 *     Scheduler, allocate_slots: a request with n tokens owns ceil(n/16) blocks;
 *     Run forward pass: slot_mapping is built while preparing inputs; all
 *       sequences are flattened into one super-sequence without padding and
 *       each token attends only to its own sequence;
 *     Prefix Caching: the forward pass fills the allocated blocks with KVs.
 *   "Serving models at scale with vLLM",
 *     PagedAttention: a block table lists a request's blocks in order;
 *     Chunked prefill: a later chunk reads the earlier chunks' KV from the
 *       cache; decodes come first in the step, then prefill chunks.
 *   "LLM Serving Frameworks #1: Deep Dive into vLLM", section 4: several
 *     block tables may name the same physical block (shared prefix).
 *
 * Conventions for every call:
 *   - All tensors are contiguous, row-major, in device memory owned by the
 *     caller.  The library allocates nothing and keeps no pointer after the
 *     call returns.  Work is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and runs asynchronously: the call never
 *     synchronises the device.
 *   - Shapes:  q, out        [num_tokens][num_q_heads][head_size]
 *              k, v          [num_tokens][num_kv_heads][head_size]
 *              k_cache, v_cache [num_blocks][block_size][num_kv_heads][head_size]
 *     Element type is layout->dtype, except the caches: layout->cache_dtype.
 *   - Return value: PA_OK, or an error code with a message for
 *     pa_last_error().  Argument errors are found on the host before anything
 *     is launched.  Values that live in device memory (slots, block ids,
 *     lengths) are checked by the kernels: an offending access is skipped and
 *     a bit is OR-ed into *status (if status is not NULL); nothing traps.
 *     The caller reads *status whenever it likes (it is a device int32).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = 1,      /* bad argument (null pointer, bad size, misalignment) */
  PA_ERR_UNSUPPORTED = 2,  /* valid but not built: head_size, GQA group, block_size */
  PA_ERR_CUDA = 3          /* a CUDA runtime call or launch failed */
} pa_status;

typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

/* Bits the kernels OR into the optional device status word. */
#define PA_DEV_SLOT_RANGE 1   /* slot >= num_blocks*block_size: that token's write skipped */
#define PA_DEV_BLOCK_RANGE 2  /* a used block-table entry outside [0,num_blocks): read as zeros */
#define PA_DEV_QSL 4          /* query_start_loc not 0-based, decreasing, or not ending at num_tokens */
#define PA_DEV_LENGTHS 8      /* q_len < 1, q_len > seq_len, or a host upper bound exceeded */
#define PA_DEV_CAPACITY 16    /* the workspace was sized for a smaller step */
#define PA_DEV_TIMEOUT 32     /* a tensor-core wait gave up; that kernel stopped early */

/* Model-side shape of the KV cache. Supported: block_size 16; head_size 64
 * or 128; num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 *   dtype        element type of q, out and the new k, v: PA_F32 or PA_BF16.
 *   cache_dtype  element type of k_cache / v_cache: equal to dtype, or
 *                PA_FP8_E4M3 with dtype PA_BF16 (8-bit KV; "Serving models at
 *                scale with vLLM", section Your model is too big: KV data can
 *                be kept at 8-bit precision).  An FP8 element holds
 *                code = E4M3(x / scale) (float32 division, round to nearest
 *                even, saturating at +-448) and stands for code * scale.
 *   k_scale, v_scale  the per-tensor scales of an FP8 cache (finite, > 0);
 *                ignored otherwise. */
typedef struct {
  int num_q_heads;
  int num_kv_heads;
  int head_size;
  int block_size;
  int num_blocks;
  pa_dtype dtype;
  pa_dtype cache_dtype;
  float k_scale;
  float v_scale;
} pa_layout;

/*
 * reshape_and_cache: for every t < num_tokens with s = slot_mapping[t] >= 0,
 * copy k[t] and v[t] (num_kv_heads x head_size elements each, bits unchanged)
 * to k_cache[s / block_size][s % block_size] and the same row of v_cache.
 * With an FP8 cache the rows are quantised on the way (see pa_layout).
 * Tokens with s < 0 are skipped.  Slots must be distinct (two tokens writing
 * one slot race).  s >= num_blocks*block_size sets PA_DEV_SLOT_RANGE.
 *
 *   k, v          device, [num_tokens][num_kv_heads][head_size], 16-byte aligned
 *   slot_mapping  device int64 [num_tokens]
 *   k_cache, v_cache  device, layout above, 16-byte aligned; written in place
 *   status        device int32 or NULL
 *   stream        cudaStream_t
 * num_tokens == 0 is a no-op.
 */
int pa_cache_write(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                   void* k_cache, void* v_cache, const pa_layout* layout, int32_t* status,
                   void* stream);

/*
 * Bytes of device workspace pa_forward needs for a step with at most
 * num_seqs requests, num_tokens new tokens and max_seq_len KV tokens per
 * request.  Returns 0 on bad arguments (see pa_last_error).
 */
size_t pa_forward_workspace_size(const pa_layout* layout, int num_seqs, int num_tokens,
                                 int max_seq_len);

/*
 * Attention for the flattened step.  Request r owns rows
 * query_start_loc[r] .. query_start_loc[r+1]-1 of q/out (L = its q_len) and
 * S = seq_lens[r] KV tokens, this step's included (they must already be in
 * the cache, see pa_cache_write).  Row j of the request sits at position
 * S - L + j and attends causally to positions 0 .. S - L + j; position p is
 * row p % block_size of block block_tables[r * max_blocks_per_seq + p / block_size].
 * q head h reads kv head h / (num_q_heads / num_kv_heads).
 *
 *   out[t][h] = sum_p softmax_p(scale * q[t][h] . K[p]) V[p]
 *
 * computed with fp32 accumulation and written in layout->dtype.
 *
 *   block_tables     device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                    ceil(S/block_size) are never read
 *   seq_lens         device int32 [num_seqs]
 *   query_start_loc  device int32 [num_seqs + 1], 0-based, nondecreasing,
 *                    ending at num_tokens
 *   max_query_len, max_seq_len  host upper bounds of q_len and seq_len (no
 *                    device-to-host copy is made); a request above them sets
 *                    PA_DEV_LENGTHS and is skipped
 *   workspace        device scratch of at least
 *                    pa_forward_workspace_size(layout, num_seqs, num_tokens,
 *                    max_seq_len) bytes, 256-byte aligned; its contents need no
 *                    initialisation and are overwritten
 *   out              device, [num_tokens][num_q_heads][head_size]
 * Rows of skipped requests are left unwritten.
 *
 * The call's first kernel reads seq_lens and query_start_loc as soon as it
 * starts, which may be while the kernel before it in `stream` still runs, if
 * that kernel lets dependent launches start early (pa_cache_write does;
 * ordinary kernels, copies and event waits do not).  Such a kernel must not
 * write them.  Everything else pa_forward reads is read only after the
 * previous kernel has finished.
 *
 * Streams: everything is ordered on `stream`.  When the step can hold bf16
 * chunks of at least 16 tokens (max_query_len >= 16), their tensor-core
 * kernel runs on a library side stream forked from `stream` after the
 * planning kernel and joined back before the call returns, so it overlaps
 * the decode kernel (unless pa_set_prefill_overlap(0) asked for one stream).
 * The side stream and its two events are created once
 * per host thread and device, on the first such call (they hold no device
 * memory); make that first call before capturing `stream` into a CUDA graph.
 * A captured step records the fork and join as parallel graph branches.
 */
int pa_forward(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int max_blocks_per_seq,
               const int32_t* seq_lens, const int32_t* query_start_loc,
               int num_seqs, int num_tokens, int max_query_len, int max_seq_len,
               float scale, void* out, void* workspace, size_t workspace_bytes,
               const pa_layout* layout, int32_t* status, void* stream);

/*
 * Profiling aid (no counterpart on the pages).  With start and stop set to
 * caller-owned cudaEvent_t handles, every later pa_forward call on this
 * thread records `start` on its stream just before the decode-attention
 * kernel and `stop` just after it, so the caller can time that kernel alone.
 * The events sit between the planning kernel and the decode kernel, so while
 * they are set the decode kernel cannot start before the plan has finished
 * (its launch no longer overlaps the plan's tail): time whole steps with them
 * off.  pa_set_profile_events(NULL, NULL) turns this off.  Always returns PA_OK.
 */
int pa_set_profile_events(void* start, void* stop);

/*
 * Profiling aid (no counterpart on the pages): the same for the tensor-core
 * prefill kernel.  `start` and `stop` are recorded just before and after it
 * on the stream it is launched on (the side stream, or `stream` when the
 * overlap is off, see pa_set_prefill_overlap).  NULL, NULL turns this off.
 * Always returns PA_OK.
 */
int pa_set_prefill_profile_events(void* start, void* stop);

/*
 * Scheduling choice (no counterpart on the pages).  on != 0 (the default):
 * the tensor-core prefill kernel of a step runs on the library side stream
 * beside the decode kernel (see pa_forward).  on == 0: it runs on `stream`
 * between the planning kernel and the decode kernel, and no side stream is
 * used.  Results are bit-identical either way (the kernels write disjoint
 * output rows).  Applies to later pa_forward calls on this host thread.
 * Always returns PA_OK.
 */
int pa_set_prefill_overlap(int on);

/*
 * pa_forward without a caller-provided workspace, for callers that cannot
 * allocate device memory.  The pages have no counterpart; this is a
 * convenience of this library.  Who needs it: a serving engine that, at
 * start-up, claimed nearly all free GPU memory for its KV-block pool (so a
 * later cudaMalloc may fail), a plugin whose host framework owns all device
 * memory and hands it no allocator, or a step loop that cannot afford the
 * device synchronisation cudaMalloc/cudaFree may cause.
 *
 * Same arguments and results as pa_forward, minus workspace/workspace_bytes.
 * The scratch is one file-scope device array of PA_STATIC_SCRATCH_BYTES
 * inside the library: every GPU that loads the library holds it until the
 * process exits.  A step whose pa_forward_workspace_size exceeds that is
 * rejected with PA_ERR_INVALID before anything is launched.  The call makes
 * no cudaMalloc/cudaFree or other device-memory allocation (a step with
 * prefill chunks may, on its first call, create pa_forward's side stream and
 * events, which hold no device memory).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture starts on the device.  The address is kept for
 * the life of the process: after cudaDeviceReset on a device the array may
 * live elsewhere and the kept address is stale, so a process that resets a
 * device must not call this entry point on it again.  All calls share the one
 * array and each call re-initialises what it needs, but calls whose work
 * overlaps on the GPU (other streams, other threads) race on it: order them.
 */
#define PA_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
int pa_forward_noalloc(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* seq_lens, const int32_t* query_start_loc,
                       int num_seqs, int num_tokens, int max_query_len, int max_seq_len,
                       float scale, void* out, const pa_layout* layout, int32_t* status,
                       void* stream);

/* Message of the last failing call on this thread ("" if none). */
const char* pa_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
