"""pa_forward_noalloc: attention with the library's built-in device scratch,
for callers that cannot allocate device memory (for example a serving
engine that gave nearly all free GPU memory to its KV pool at start-up).

The GPU test calls the entry point through the C ABI on three different
steps in a row, the last with a chunk on the tensor-core prefill path, and
checks each result against pa_forward with a caller workspace on the same
inputs.  The later calls show that what an earlier call left in the shared
scratch does not leak into the next result.  This
file is collected last so that a run stopping at its first failure has run
every other test before it."""
import ctypes

import pytest
import torch

import paged_kv_attention_04_gb300 as P
from paged_kv_attention_04_gb300 import workloads as W

from helpers import TOL

PA_STATIC_SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_04_gb300 import build
    build.build()
    return P.lib()


def _call_noalloc(lib, st, lay, out, status):
    return lib.pa_forward_noalloc(
        st.q.data_ptr(), st.k_cache.data_ptr(), st.v_cache.data_ptr(), st.block_tables.data_ptr(),
        int(st.block_tables.shape[1]), st.seq_lens.data_ptr(), st.query_start_loc.data_ptr(),
        st.spec.num_seqs, st.spec.num_tokens, st.max_query_len, st.max_seq_len,
        ctypes.c_float(st.scale), out.data_ptr(), ctypes.byref(lay), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_oversized_step_is_rejected_before_any_launch(lib):
    lay = P.make_layout(32, 8, 128, 30000, torch.bfloat16)
    need = P.pa_forward_workspace_size(lay, 1024, 1024, 8192)
    assert need > PA_STATIC_SCRATCH_BYTES
    rc = lib.pa_forward_noalloc(256, 256, 256, 256, 512, 256, 256, 1024, 1024, 1, 8192,
                                ctypes.c_float(0.1), 256, ctypes.byref(lay), None, None)
    assert rc == P.PA_ERR_INVALID
    assert "scratch" in P.last_error()


@pytest.mark.gpu
def test_noalloc_matches_pa_forward_on_calls_in_a_row(lib):
    specs = [
        # decodes that split over several KV blocks, plus a multi-token chunk
        W.custom_spec("noalloc-a", "bf16", 32, 8, 128, [1, 1, 6, 1], [900, 17, 70, 2500], seed=41),
        # different shape and head layout: the scratch is reused with new contents
        W.custom_spec("noalloc-b", "bf16", 16, 2, 64, [1, 3, 1], [3000, 40, 128], seed=42),
        # a 40-token chunk on the tensor-core prefill path (its work list, counter
        # and KV-split partial states in the scratch), after calls that left
        # other contents there
        W.custom_spec("noalloc-c", "bf16", 32, 8, 128, [1, 40, 1], [600, 340, 2100], seed=43),
    ]
    for spec in specs:
        st = W.make_step(spec, device="cuda")
        lay = P.layout_of(st.k_cache, spec.num_q_heads)
        assert P.pa_forward_workspace_size(lay, spec.num_seqs, spec.num_tokens,
                                           st.max_seq_len) <= PA_STATIC_SCRATCH_BYTES
        P.pa_cache_write(st.k, st.v, st.slot_mapping, st.k_cache, st.v_cache, lay)
        ws = P.alloc_workspace(lay, spec.num_seqs, spec.num_tokens, st.max_seq_len)
        ref = torch.full_like(st.q, float("nan"))
        P.pa_forward(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                     st.query_start_loc, st.max_query_len, st.max_seq_len, st.scale, ref, ws, lay)
        out = torch.full_like(st.q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _call_noalloc(lib, st, lay, out, status)
        assert rc == P.PA_OK, P.last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert not ref.isnan().any() and not out.isnan().any()
        atol, rtol = TOL["bf16"]
        err = (out.double() - ref.double()).abs()
        assert bool((err <= atol + rtol * ref.double().abs()).all()), float(err.max())
