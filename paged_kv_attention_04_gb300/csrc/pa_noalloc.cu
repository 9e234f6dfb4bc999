// pa_forward_noalloc: pa_forward with the library's own device scratch, for
// callers that cannot allocate device memory (see include/pa.h).
//
// The scratch is one file-scope device array.  In host code its name is only
// a host-side stand-in, so its device address is looked up once per device
// (with that device current) and that address is what pa_forward receives.
// Every workspace word pa_forward relies on is rewritten by its plan kernel
// at the start of each call, so nothing needs clearing here; calls that
// overlap on the GPU share the array and race.
#include <cstdio>
#include <mutex>
#include <string>

#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_pa_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_pa_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return pa::set_last_error(PA_ERR_CUDA, (std::string("cudaGetDevice: ") +
                                            cudaGetErrorString(e)).c_str());
  if (dev < 0 || dev >= kMaxDevices)
    return pa::set_last_error(PA_ERR_CUDA, "device ordinal out of range for the static scratch");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pa_scratch);
    if (e != cudaSuccess || !p)
      return pa::set_last_error(PA_ERR_CUDA, (std::string("cudaGetSymbolAddress(scratch): ") +
                                              cudaGetErrorString(e)).c_str());
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_forward_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* seq_lens, const int32_t* query_start_loc,
                                  int num_seqs, int num_tokens, int max_query_len,
                                  int max_seq_len, float scale, void* out,
                                  const pa_layout* layout, int32_t* status, void* stream) {
  if (num_seqs == 0 || num_tokens == 0)
    return pa_forward(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                      query_start_loc, num_seqs, num_tokens, max_query_len, max_seq_len, scale,
                      out, nullptr, 0, layout, status, stream);
  const size_t need = pa_forward_workspace_size(layout, num_seqs, num_tokens, max_seq_len);
  if (need == 0) return PA_ERR_INVALID;  // message already set
  if (need > PA_STATIC_SCRATCH_BYTES) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "step needs %zu bytes of scratch; the built-in scratch holds %zu "
             "(use pa_forward with a caller workspace)",
             need, static_cast<size_t>(PA_STATIC_SCRATCH_BYTES));
    return pa::set_last_error(PA_ERR_INVALID, buf);
  }
  void* ws = nullptr;
  if (int rc = scratch_address(&ws)) return rc;
  return pa_forward(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                    query_start_loc, num_seqs, num_tokens, max_query_len, max_seq_len, scale, out,
                    ws, PA_STATIC_SCRATCH_BYTES, layout, status, stream);
}
