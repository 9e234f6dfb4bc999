"""Paged-KV attention for one continuous-batching step on GB300 (sm_103a).

The computation lives in libpa.so (hand-written CUDA kernels behind a C ABI,
declared in include/pa.h); `binding` exposes the same calls on torch tensors.
"""
from .binding import (PA_BF16, PA_DEV_BLOCK_RANGE, PA_DEV_CAPACITY, PA_DEV_LENGTHS, PA_DEV_QSL,
                      PA_DEV_SLOT_RANGE, PA_DEV_TIMEOUT, PA_ERR_CUDA, PA_ERR_INVALID,
                      PA_ERR_UNSUPPORTED, PA_F32, PA_FP8_E4M3, PA_OK, PaError, alloc_workspace,
                      last_error, layout_of, lib, make_layout, pa_cache_write, pa_forward,
                      pa_forward_noalloc, pa_forward_workspace_size, pa_layout,
                      pa_set_prefill_overlap, pa_set_prefill_profile_events,
                      pa_set_profile_events)

__all__ = ["PA_BF16", "PA_DEV_BLOCK_RANGE", "PA_DEV_CAPACITY", "PA_DEV_LENGTHS", "PA_DEV_QSL",
           "PA_DEV_SLOT_RANGE", "PA_DEV_TIMEOUT", "PA_ERR_CUDA", "PA_ERR_INVALID",
           "PA_ERR_UNSUPPORTED", "PA_F32", "PA_FP8_E4M3", "PA_OK", "PaError", "alloc_workspace",
           "last_error", "layout_of", "lib", "make_layout", "pa_cache_write", "pa_forward",
           "pa_forward_noalloc", "pa_forward_workspace_size", "pa_layout",
           "pa_set_prefill_overlap", "pa_set_prefill_profile_events", "pa_set_profile_events"]
