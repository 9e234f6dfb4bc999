"""Malformed device-resident inputs are caught by the kernels' own checks:
the offending access is skipped and a status bit is set; nothing traps and
the rest of the step is still computed."""
import numpy as np
import pytest
import torch

import paged_kv_attention_04_gb300 as P
from paged_kv_attention_04_gb300 import workloads as W

from helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_attention_04_gb300 import build
    build.build()
    P.lib()


def _step():
    spec = W.custom_spec("err", "bf16", 8, 2, 64, [1, 1, 3], [20, 40, 30], seed=3)
    return W.make_step(spec)


def _forward(st, **over):
    lay = P.layout_of(st.k_cache, st.spec.num_q_heads)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = P.alloc_workspace(lay, st.spec.num_seqs, st.spec.num_tokens, st.max_seq_len)
    out = torch.full_like(st.q, float("nan"))
    args = dict(seq_lens=st.seq_lens, qsl=st.query_start_loc, bt=st.block_tables,
                maxq=st.max_query_len, maxs=st.max_seq_len)
    args.update(over)
    P.pa_forward(st.q, st.k_cache, st.v_cache, args["bt"], args["seq_lens"], args["qsl"],
                 args["maxq"], args["maxs"], st.scale, out, ws, lay, status)
    torch.cuda.synchronize()
    return out, int(status.item())


def test_slot_out_of_range_is_skipped_and_flagged():
    st = _step().to("cuda")
    kc, vc = st.k_cache.clone(), st.v_cache.clone()
    lay = P.layout_of(kc, 8)
    slots = st.slot_mapping.clone()
    slots[1] = st.num_blocks * 16 + 5
    slots[2] = -1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pa_cache_write(st.k, st.v, slots, kc, vc, lay, status)
    torch.cuda.synchronize()
    assert int(status.item()) & P.PA_DEV_SLOT_RANGE
    flat = kc.view(-1, 2, 64)
    assert torch.equal(flat[slots[0]], st.k[0])
    assert torch.equal(flat[slots[3]], st.k[3])
    # skipped tokens left their slots untouched (still NaN)
    assert flat[st.slot_mapping[1]].isnan().all() and flat[st.slot_mapping[2]].isnan().all()


def test_block_id_out_of_range_is_flagged():
    st = _step().to("cuda")
    bt = st.block_tables.clone()
    bt[1, 0] = st.num_blocks + 1000
    out, status = _forward(st, bt=bt)
    assert status & P.PA_DEV_BLOCK_RANGE


def test_bad_query_start_loc_schedules_nothing():
    st = _step().to("cuda")
    qsl = st.query_start_loc.clone()
    qsl[-1] = qsl[-1] - 1
    out, status = _forward(st, qsl=qsl)
    assert status & P.PA_DEV_QSL
    assert out.isnan().all()


def test_length_errors_skip_only_that_request():
    cpu = _step()
    st = cpu.to("cuda")
    # write this step's KV first so the valid requests can be checked
    lay = P.layout_of(st.k_cache, 8)
    P.pa_cache_write(st.k, st.v, st.slot_mapping, st.k_cache, st.v_cache, lay)
    seq = st.seq_lens.clone()
    seq[2] = 2                       # q_len 3 > seq_len 2
    out, status = _forward(st, seq_lens=seq)
    assert status & P.PA_DEV_LENGTHS
    assert out[2:].isnan().all()
    ref, _, _ = run_oracle(cpu)
    assert_close(out[:2], ref[:2], "bf16", "valid requests")
    # a request longer than the host bound is skipped too
    out, status = _forward(st, maxs=39)
    assert status & P.PA_DEV_LENGTHS
    assert out[1].isnan().all()
    assert_close(out[0], ref[0], "bf16", "request 0")
