"""A step (pa_cache_write + pa_forward) captured in a CUDA graph replays to the
same bits as eager calls, with new inputs copied into the captured buffers.

"Serving models at scale with vLLM", section CUDA graphs: the forward pass
is recorded once per batch shape and replayed, which removes launch gaps
(decode steps gain most).  Capture needs the calls to make no host
synchronisation and no allocation; the library's per-device set-up happens
on the first eager call, so one eager call precedes the capture."""
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


def _step_fn(st, lay, ws, out, status):
    def fn():
        P.pa_cache_write(st.k, st.v, st.slot_mapping, st.k_cache, st.v_cache, lay, status)
        P.pa_forward(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                     st.query_start_loc, st.max_query_len, st.max_seq_len, st.scale, out, ws, lay,
                     status)
    return fn


@pytest.mark.parametrize("mixed", [False, True])
def test_graph_replay_matches_eager_and_oracle(mixed):
    if mixed:
        spec = W.custom_spec("graph-mixed", "bf16", 32, 8, 128, [1, 1, 3, 40], [700, 20, 90, 300],
                             seed=51)
    else:
        spec = W.custom_spec("graph-decode", "bf16", 32, 4, 64, [1] * 6, [5, 16, 17, 400, 1500, 64],
                             seed=52)
    cpu = W.make_step(spec)
    st = cpu.to("cuda")
    lay = P.layout_of(st.k_cache, spec.num_q_heads)
    ws = P.alloc_workspace(lay, spec.num_seqs, spec.num_tokens, st.max_seq_len)
    out = torch.full_like(st.q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k0, v0 = st.k_cache.clone(), st.v_cache.clone()
    fn = _step_fn(st, lay, ws, out, status)

    fn()  # eager: per-device set-up happens here, before any capture
    torch.cuda.synchronize()
    eager1 = out.clone()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g):
            fn()
    torch.cuda.current_stream().wait_stream(s)

    # replay 1: same inputs, restored caches
    st.k_cache.copy_(k0)
    st.v_cache.copy_(v0)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager1.view(torch.int16))

    # replay 2: new q and new K/V for the step's tokens, copied into the captured buffers
    gen = torch.Generator(device="cuda").manual_seed(7)
    new_q = torch.randn(st.q.shape, generator=gen, device="cuda").to(st.q.dtype)
    new_k = torch.randn(st.k.shape, generator=gen, device="cuda").to(st.k.dtype)
    new_v = torch.randn(st.v.shape, generator=gen, device="cuda").to(st.v.dtype)
    st.q.copy_(new_q)
    st.k.copy_(new_k)
    st.v.copy_(new_v)
    st.k_cache.copy_(k0)
    st.v_cache.copy_(v0)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    graph2 = out.clone()
    assert int(status.item()) == 0

    st.k_cache.copy_(k0)
    st.v_cache.copy_(v0)
    out.fill_(float("nan"))
    fn()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), graph2.view(torch.int16))

    cpu.q, cpu.k, cpu.v = new_q.cpu(), new_k.cpu(), new_v.cpu()
    ref, _, _ = run_oracle(cpu)
    assert_close(graph2, ref, "bf16", "graph replay")
