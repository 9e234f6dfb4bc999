"""fp64 CPU oracle for the paged-KV attention step.

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's
CPU-baseline leg use it.  The product path (the CUDA library and its Python
binding) never imports it.
"""
from .paged_attention import (blocks_needed, block_bytes, slot_of, widen, validate_step,
                              cache_write, gather_request_kv, paged_attention,
                              paged_attention_rows, within_tolerance, error_report)

__all__ = ["blocks_needed", "block_bytes", "slot_of", "widen", "validate_step", "cache_write",
           "gather_request_kv", "paged_attention", "paged_attention_rows", "within_tolerance",
           "error_report"]
