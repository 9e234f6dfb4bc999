"""FP8 (E4M3) KV cache: the quantising slot write matches the oracle bit for
bit, and attention over the 8-bit cache matches the fp64 oracle over the
dequantised cache within the bf16 tolerance (both sides see the same
quantised values)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
import paged_kv_attention_04_gb300 as P
from paged_kv_attention_04_gb300 import workloads as W

from helpers import assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_attention_04_gb300 import build
    build.build()
    P.lib()


def _pool_codes(cache_bf16, scale):
    """History pool as E4M3 codes, by torch's float8 cast (input preparation)."""
    x = cache_bf16.float() / scale
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def _run(spec, k_scale, v_scale):
    cpu = W.make_step(spec)
    kc0 = _pool_codes(cpu.k_cache, k_scale)
    vc0 = _pool_codes(cpu.v_cache, v_scale)
    st = cpu.to("cuda")
    kc, vc = kc0.cuda(), vc0.cuda()
    lay = P.layout_of(kc, spec.num_q_heads, k_scale=k_scale, v_scale=v_scale)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pa_cache_write(st.k, st.v, st.slot_mapping, kc, vc, lay, status)
    ws = P.alloc_workspace(lay, spec.num_seqs, spec.num_tokens, st.max_seq_len)
    out = torch.full_like(st.q, float("nan"))
    P.pa_forward(st.q, kc, vc, st.block_tables, st.seq_lens, st.query_start_loc,
                 st.max_query_len, st.max_seq_len, st.scale, out, ws, lay, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # oracle: quantising slot write, then attention over the dequantised cache
    rk, rv = fp8.cache_write_fp8(oracle.widen(bits(cpu.k)), oracle.widen(bits(cpu.v)),
                                 cpu.slot_mapping.numpy(), kc0.numpy(), vc0.numpy(),
                                 k_scale, v_scale)
    assert np.array_equal(kc.cpu().numpy(), rk)
    assert np.array_equal(vc.cpu().numpy(), rv)
    ref = oracle.paged_attention(bits(cpu.q), fp8.dequantize(rk, k_scale), fp8.dequantize(rv, v_scale),
                                 cpu.block_tables.numpy(), spec.seq_lens, cpu.query_start_loc.numpy(),
                                 cpu.scale, spec.num_kv_heads)
    return assert_close(out, ref, "bf16", spec.name)


def test_llama3_8b_decode_fp8():
    _run(W.spec_llama3_8b_decode(), 0.01, 0.01)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_random_shapes_fp8(D, G):
    spec = W.custom_spec(f"fp8-{D}-{G}", "bf16", 2 * G, 2, D, [1, 1, 3, 1, 20],
                         [1, 17, 40, 700, 300], seed=70 + D + G)
    # scale 0.005 makes |x| > 2.24 saturate at 448: the saturating path is exercised
    _run(spec, 0.005, 0.02)


def test_fp8_layout_checks():
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(P.PaError):
        P.pa_forward_workspace_size(P.layout_of(kc, 4, dtype=torch.float32), 1, 1, 16)
    with pytest.raises(P.PaError):
        P.pa_forward_workspace_size(P.layout_of(kc, 4, k_scale=0.0), 1, 1, 16)


@pytest.mark.parametrize("D", [64, 128])
def test_fp8_chunks_on_tensor_cores(D):
    """Chunks of 17-300 tokens over an 8-bit cache take the tensor-core prefill
    kernel (codes widened to f16 in shared memory); with fewer units than SMs
    their KV is split into pieces that are merged.  Checked against the oracle
    over the dequantised cache."""
    spec = W.custom_spec(f"fp8-chunks-{D}", "bf16", 8, 2, D, [1, 300, 1, 64, 17],
                         [700, 2300, 40, 64, 900], seed=77 + D)
    _run(spec, 0.01, 0.02)


def test_fp8_short_chunk_long_prior():
    """A 16-token chunk after ~6000 tokens of context over an 8-bit cache: one
    unit per kv head, cut into many pieces (one round over the SMs), each
    piece's tiles widened by the softmax warps, merged by the last piece."""
    spec = W.custom_spec("fp8-long-prior", "bf16", 8, 2, 128, [16, 1], [6016, 300], seed=71)
    _run(spec, 0.01, 0.02)


def test_fp8_mixed_step():
    """The mixed continuous-batching step (192 decodes, two 512-token chunks)
    over an 8-bit cache: decode and few-token kernels read codes, the chunks
    run on the tensor cores."""
    _run(W.spec_mixed_step(), 0.01, 0.01)


@pytest.mark.parametrize("D,G", [(64, 8), (64, 2), (128, 1)])
def test_fp8_long_chunks(D, G):
    """Chunks of 40-300 tokens over 1000-3000 keys (up to 24 KV tiles a unit,
    several units per CTA) over an 8-bit cache: K codes run two tiles ahead
    in staging buffers, V codes land in place in the V buffers, across tiles
    and units, and the last tile's ragged block is zeroed."""
    spec = W.custom_spec(f"fp8-long-{D}-{G}", "bf16", 2 * G, 2, D, [300, 1, 129, 40],
                         [3000, 77, 1001, 1500], seed=90 + D + G)
    _run(spec, 0.01, 0.02)


def test_fp8_chunked_schedule_sampled():
    """The chunked schedule (152 units of ~30 KV tiles cut into equal chunks)
    over an 8-bit cache: the quantising write bit for bit, attention on
    sampled rows against the oracle over the dequantised cache."""
    L, prior, Hkv, D = 19 * 128, 3000, 8, 128
    spec = W.custom_spec("fp8-chunked", "bf16", Hkv, Hkv, D, [L], [prior + L], seed=451)
    cpu = W.make_step(spec)
    ks, vs = 0.01, 0.02
    kc0, vc0 = _pool_codes(cpu.k_cache, ks), _pool_codes(cpu.v_cache, vs)
    st = cpu.to("cuda")
    kc, vc = kc0.cuda(), vc0.cuda()
    lay = P.layout_of(kc, spec.num_q_heads, k_scale=ks, v_scale=vs)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pa_cache_write(st.k, st.v, st.slot_mapping, kc, vc, lay, status)
    ws = P.alloc_workspace(lay, spec.num_seqs, spec.num_tokens, st.max_seq_len)
    out = torch.full_like(st.q, float("nan"))
    P.pa_forward(st.q, kc, vc, st.block_tables, st.seq_lens, st.query_start_loc,
                 st.max_query_len, st.max_seq_len, st.scale, out, ws, lay, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rk, rv = fp8.cache_write_fp8(oracle.widen(bits(cpu.k)), oracle.widen(bits(cpu.v)),
                                 cpu.slot_mapping.numpy(), kc0.numpy(), vc0.numpy(), ks, vs)
    assert np.array_equal(kc.cpu().numpy(), rk) and np.array_equal(vc.cpu().numpy(), rv)
    nb = oracle.blocks_needed(prior + L)
    bt = cpu.block_tables.numpy()[0, :nb]
    rows = [(j, g) for g in range(Hkv) for j in (0, 127, 128, L // 2, L - 1)]
    ref = oracle.paged_attention_rows(bits(cpu.q), fp8.dequantize(rk, ks)[bt], fp8.dequantize(rv, vs)[bt],
                                      np.arange(nb)[None, :], spec.seq_lens, np.array([0, L]),
                                      cpu.scale, Hkv, rows)
    got = torch.stack([out[t, h] for t, h in rows])
    assert_close(got, ref, "bf16", spec.name)
