"""GPU parity: libpa against the fp64 oracle on the same seeded inputs.

Cache writes must match bit for bit (the whole cache, so untouched slots are
checked too).  Attention outputs must be finite and meet, with (atol, rtol) =
(1e-2, 2e-2) for bf16 and (1e-5, 1e-5) for fp32: |gpu - oracle| <= atol +
rtol |oracle| per element, max-abs error <= atol, and max-rel error <= rtol
over the elements with |oracle| at or above a stated floor (helpers.assert_close).
Every launch goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_04_gb300 as P
from paged_kv_attention_04_gb300 import workloads as W

from helpers import assert_close, bits, raw_bits, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_attention_04_gb300 import build
    build.build()
    P.lib()


def _full_parity(step_cpu):
    step = step_cpu.to("cuda")
    out, kc, vc, status = run_gpu(step)
    assert status == 0
    ref, rkc, rvc = run_oracle(step_cpu)
    assert np.array_equal(raw_bits(kc), rkc.view(np.uint32) if rkc.dtype == np.float32 else rkc)
    assert np.array_equal(raw_bits(vc), rvc.view(np.uint32) if rvc.dtype == np.float32 else rvc)
    return assert_close(out, ref, step_cpu.spec.dtype, step_cpu.spec.name)


@pytest.mark.parametrize("name", ["tiny_decode_f32", "tinyllama_decode", "llama3_8b_decode",
                                  "mixed_step"])
def test_config_full_parity(name):
    _full_parity(W.make_config(name))


def test_long_context_sampled_parity():
    """Long-context decode at full size (a ~9 GB pool): the whole cache write
    is checked bit for bit; attention on 128 rows the oracle evaluates one by
    one, one q head of every kv head of every request."""
    spec = W.spec_long_context_decode()
    step = W.make_step(spec, device="cuda")
    out, kc, vc, status = run_gpu(step)
    assert status == 0
    slots = step.slot_mapping
    # written rows hold the new tokens' bits; every other row is unchanged
    NBS = step.num_blocks * 16
    for cache, orig, new in ((kc, step.k_cache, step.k), (vc, step.v_cache, step.v)):
        flat = cache.view(NBS, -1).view(torch.int16)
        assert torch.equal(flat[slots], new.reshape(len(slots), -1).view(torch.int16))
        restored = flat.clone()
        restored[slots] = orig.view(NBS, -1).view(torch.int16)[slots]
        assert torch.equal(restored, orig.view(NBS, -1).view(torch.int16))
        del restored
    # oracle on every request and every kv head (one of its q heads, rotating
    # through the group), over a private copy of each request's blocks
    bt = step.block_tables.cpu().numpy()
    S_all = spec.seq_lens
    G = spec.num_q_heads // spec.num_kv_heads
    checked = 0
    for r in range(spec.num_seqs):
        S = int(S_all[r])
        nb = oracle.blocks_needed(S)
        blocks = torch.from_numpy(bt[r, :nb].astype(np.int64)).cuda()
        mk = bits(step.k_cache[blocks])
        mv = bits(step.v_cache[blocks])
        pos = S - 1
        slot = (pos // 16) * 16 + pos % 16
        mk, mv = oracle.cache_write(bits(step.k[r:r + 1]), bits(step.v[r:r + 1]),
                                    np.array([slot]), mk, mv)
        rows = [(0, g * G + (r + g) % G) for g in range(spec.num_kv_heads)]
        ref = oracle.paged_attention_rows(bits(step.q[r:r + 1]), mk, mv, np.arange(nb)[None, :],
                                          np.array([S]), np.array([0, 1]), step.scale,
                                          spec.num_kv_heads, rows)
        got = torch.stack([out[r, h] for _, h in rows])
        assert_close(got, ref, "bf16", f"long-context r={r} S={S}")
        checked += len(rows)
        del mk, mv
    assert checked == spec.num_seqs * spec.num_kv_heads


def test_long_prefill_chunk_sampled_parity():
    """One 2048-token chunk over 8192 keys (the tensor-core kernel's steady
    state, as bench.py times it): the whole cache write is checked bit for
    bit, attention on sampled (token, head) rows that the oracle evaluates
    one by one (first and last rows of query tiles, every kv head)."""
    spec = W.spec_long_prefill_chunk()
    step = W.make_step(spec, device="cuda")
    out, kc, vc, status = run_gpu(step)
    assert status == 0
    nb = oracle.blocks_needed(int(spec.seq_lens[0]))
    blocks = torch.from_numpy(step.block_tables.cpu().numpy()[0, :nb].astype(np.int64)).cuda()
    mk, mv = oracle.cache_write(bits(step.k), bits(step.v), step.slot_mapping.cpu().numpy(),
                                bits(step.k_cache), bits(step.v_cache))
    assert np.array_equal(bits(kc), mk) and np.array_equal(bits(vc), mv)
    rows = [(0, 0), (31, 3), (32, 4), (1023, 17), (1024, 18), (2016, 26), (2047, 31), (777, 9)]
    ref = oracle.paged_attention_rows(bits(step.q), mk[blocks.cpu().numpy()],
                                      mv[blocks.cpu().numpy()], np.arange(nb)[None, :],
                                      spec.seq_lens, np.array([0, 2048]), step.scale,
                                      spec.num_kv_heads, rows)
    got = torch.stack([out[t, h] for t, h in rows])
    assert_close(got, ref, "bf16", "long prefill chunk")


def test_long_prior_chunks_sampled_parity():
    """Short chunks late in long prompts (64 tokens after 32768, 16 after
    98304), as bench.py times them: the KV of each query tile is split into
    pieces and merged.  The whole cache write is checked bit for bit,
    attention on sampled rows of both chunks and every kv head."""
    spec = W.spec_long_prior_chunks()
    step = W.make_step(spec, device="cuda")
    out, kc, vc, status = run_gpu(step)
    assert status == 0
    mk, mv = oracle.cache_write(bits(step.k), bits(step.v), step.slot_mapping.cpu().numpy(),
                                bits(step.k_cache), bits(step.v_cache))
    assert np.array_equal(bits(kc), mk) and np.array_equal(bits(vc), mv)
    bt = step.block_tables.cpu().numpy()
    qsl = step.query_start_loc.cpu().numpy()
    G = spec.num_q_heads // spec.num_kv_heads
    for r in range(spec.num_seqs):
        S, L = int(spec.seq_lens[r]), int(spec.q_lens[r])
        nb = oracle.blocks_needed(S)
        rows = [(int(qsl[r]) + j, g * G + (j + g) % G) for g in range(spec.num_kv_heads)
                for j in (0, L // 2, L - 1)]
        ref = oracle.paged_attention_rows(bits(step.q), mk[bt[r, :nb]], mv[bt[r, :nb]],
                                          np.arange(nb)[None, :].repeat(spec.num_seqs, 0),
                                          spec.seq_lens, qsl, step.scale, spec.num_kv_heads,
                                          rows)
        got = torch.stack([out[t, h] for t, h in rows])
        assert_close(got, ref, "bf16", f"long prior chunk r={r}")


@pytest.mark.parametrize("D,G", [(64, 1), (128, 1), (64, 2), (128, 2)])
def test_chunked_schedule_sampled_parity(D, G):
    """One chunk of 19 query tiles over 3000 prior keys with 8 kv heads: 152
    units of ~30 KV tiles, which the plan cuts into equal chunks of a unit
    line (units cut at chunk boundaries become pieces merged by the last).
    The whole cache write is checked bit for bit, attention on sampled rows
    (query-tile edges and the middle, every kv head)."""
    pm = 128 // G
    L, prior, Hkv = 19 * pm, 3000, 8
    spec = W.custom_spec(f"chunked-{D}-{G}", "bf16", Hkv * G, Hkv, D, [L], [prior + L], seed=400 + D + G)
    step = W.make_step(spec, device="cuda")
    out, kc, vc, status = run_gpu(step)
    assert status == 0
    mk, mv = oracle.cache_write(bits(step.k), bits(step.v), step.slot_mapping.cpu().numpy(),
                                bits(step.k_cache), bits(step.v_cache))
    assert np.array_equal(bits(kc), mk) and np.array_equal(bits(vc), mv)
    nb = oracle.blocks_needed(prior + L)
    bt = step.block_tables.cpu().numpy()[0, :nb]
    rows = [(j, g * G + (j + g) % G) for g in range(Hkv) for j in (0, pm - 1, pm, L // 2, L - 1)]
    ref = oracle.paged_attention_rows(bits(step.q), mk[bt], mv[bt], np.arange(nb)[None, :],
                                      spec.seq_lens, np.array([0, L]), step.scale, Hkv, rows)
    got = torch.stack([out[t, h] for t, h in rows])
    assert_close(got, ref, "bf16", spec.name)


def test_prefill_runs_are_bit_identical():
    """Chunks of 16 to 1000 tokens over contexts up to 3000 keys: ~450 tensor-core
    units, several per CTA, so every hand-off between the kernel's roles is
    crossed many times, including at unit boundaries.  Three runs must give the
    same bits (the kernel has no order-dependent arithmetic), and the first must
    match the oracle."""
    spec = W.custom_spec("pf-det", "bf16", 32, 8, 128, [16, 100, 513, 40, 1000, 1],
                         [16, 700, 513, 3000, 1000, 900], seed=61)
    step_cpu = W.make_step(spec)
    step = step_cpu.to("cuda")
    outs = []
    for _ in range(3):
        out, kc, vc, status = run_gpu(step)
        assert status == 0
        outs.append(out)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    ref, _, _ = run_oracle(step_cpu)
    assert_close(outs[0], ref, "bf16", "prefill determinism case")


SHAPES = [
    # (q_lens, seq_lens): decode lengths at block edges, chunks, a 1-token prompt
    ([1, 1, 1, 1, 1, 1], [1, 15, 16, 17, 300, 1000]),
    ([3, 1, 16, 40, 1], [17, 33, 40, 300, 2]),
    ([7, 1, 25], [500, 257, 25]),
    # KV splits (at least 128 blocks = 2048 keys each) and their merge: a decode one
    # block past a split, few-token queries (2-15 rows) over long contexts
    ([1, 4, 15, 2, 1], [2049, 5000, 3000, 6100, 4096]),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_random_shapes(dtype, D, G, shape):
    q_lens, seq_lens = SHAPES[shape]
    Hkv = 2
    spec = W.custom_spec(f"rand-{dtype}-{D}-{G}-{shape}", dtype, Hkv * G, Hkv, D, q_lens, seq_lens,
                         seed=100 + shape * 17 + D + G)
    _full_parity(W.make_step(spec))


def test_many_requests_plan_passes():
    """700 requests, more than the plan kernel's CTA holds at once: its passes
    over the requests carry every list's offsets, the decode dispatch order
    (long splits in request order, short ones in the shared short-item list)
    and the prefill query tiles across passes.  Decodes (some split: longer
    than 2048 keys), few-token queries (2-15) and chunks of 16-40 tokens."""
    rng = np.random.default_rng(321)
    q_lens, seq_lens = [], []
    for i in range(700):
        kind = rng.random()
        if kind < 0.8:
            q, s = 1, int(rng.integers(1, 2600))
        elif kind < 0.95:
            q = int(rng.integers(2, 16))
            s = q + int(rng.integers(0, 2400))
        else:
            q = int(rng.integers(16, 41))
            s = q + int(rng.integers(0, 600))
        q_lens.append(q)
        seq_lens.append(s)
    spec = W.custom_spec("many-requests", "bf16", 8, 2, 64, q_lens, seq_lens, seed=322)
    _full_parity(W.make_step(spec))


def test_prefix_sharing_and_permutation_invariance():
    """Outputs are bit-identical when the physical blocks are renumbered (data
    moved with them), including blocks shared by several tables."""
    spec = W.custom_spec("perm", "bf16", 8, 2, 128, [1, 1, 1, 4], [40, 90, 200, 64],
                         shared_prefix_blocks=2, sharing=[True, True, True, False], seed=9)
    st = W.make_step(spec, device="cuda")
    out1, *_ = run_gpu(st)
    NB = st.num_blocks
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(4)).cuda()
    st2 = W.make_step(spec, device="cuda")
    st2.k_cache = torch.empty_like(st.k_cache)
    st2.v_cache = torch.empty_like(st.v_cache)
    st2.k_cache[perm] = st.k_cache
    st2.v_cache[perm] = st.v_cache
    bt = st.block_tables.long()
    st2.block_tables = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int()
    st2.slot_mapping = perm[st.slot_mapping // 16] * 16 + st.slot_mapping % 16
    out2, *_ = run_gpu(st2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_batch_invariance_and_determinism():
    spec = W.custom_spec("batch", "bf16", 32, 8, 128, [1, 5, 1, 1], [700, 64, 3000, 16], seed=21)
    st = W.make_step(spec, device="cuda")
    out, *_ = run_gpu(st)
    again, *_ = run_gpu(st)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    qsl = st.query_start_loc.tolist()
    for r in range(4):
        solo = W.custom_spec("solo", "bf16", 32, 8, 128, [spec.q_lens[r]], [spec.seq_lens[r]], seed=21)
        s1 = W.make_step(solo, device="cuda")
        s1.k_cache, s1.v_cache = st.k_cache, st.v_cache
        s1.block_tables = st.block_tables[r:r + 1].contiguous()
        s1.q = st.q[qsl[r]:qsl[r + 1]].contiguous()
        s1.k = st.k[qsl[r]:qsl[r + 1]].contiguous()
        s1.v = st.v[qsl[r]:qsl[r + 1]].contiguous()
        s1.slot_mapping = st.slot_mapping[qsl[r]:qsl[r + 1]].contiguous()
        o1, *_ = run_gpu(s1)
        assert torch.equal(o1.view(torch.int16), out[qsl[r]:qsl[r + 1]].view(torch.int16))


def test_chunked_prefill_matches_whole_prompt():
    """A prompt run as chunks (each written, then attended) matches the whole
    prompt run at once, within tolerance of the oracle."""
    n, chunks = 600, (256, 256, 88)
    spec = W.custom_spec("whole", "bf16", 16, 4, 128, [n], [n], seed=31)
    st = W.make_step(spec, device="cuda")
    whole, *_ = run_gpu(st)
    kc, vc = st.k_cache.clone(), st.v_cache.clone()
    lay = P.layout_of(kc, 16)
    done, parts = 0, []
    for c in chunks:
        sl = slice(done, done + c)
        P.pa_cache_write(st.k[sl], st.v[sl], st.slot_mapping[sl], kc, vc, lay)
        sq = torch.tensor([done + c], dtype=torch.int32, device="cuda")
        qsl = torch.tensor([0, c], dtype=torch.int32, device="cuda")
        ws = P.alloc_workspace(lay, 1, c, done + c)
        o = torch.empty_like(st.q[sl])
        P.pa_forward(st.q[sl].contiguous(), kc, vc, st.block_tables, sq, qsl, c, done + c, st.scale,
                     o, ws, lay)
        parts.append(o)
        done += c
    chunked = torch.cat(parts)
    torch.cuda.synchronize()
    ref, _, _ = run_oracle(st.to("cpu"))
    assert_close(chunked, ref, "bf16", "chunked")
    assert_close(whole, ref, "bf16", "whole")


def test_empty_step_is_a_noop():
    lay = P.make_layout(8, 2, 64, 4, torch.bfloat16)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    e = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    P.pa_cache_write(e, e, torch.empty(0, dtype=torch.int64, device="cuda"), kc, kc, lay)
    torch.cuda.synchronize()
    assert int(kc.abs().sum()) == 0


PREFILL_SHAPES = [
    # q_len around the tensor-core threshold (15 -> few-token tiles, 16/17 -> tcgen05)
    ("bf16", 128, 4, [15, 16, 17], [15, 40, 17]),
    # last 128-row tile holds one position (33 = 32 + 1 positions at G = 4)
    ("bf16", 128, 4, [33, 1], [33, 90]),
    # long prior context: ~40 KV tiles of 128 tokens behind a 300-token chunk
    ("bf16", 128, 4, [300], [5000]),
    # G = 8, D = 64: 16 positions per 128-row tile
    ("bf16", 64, 8, [70, 1, 16], [1000, 50, 16]),
    # G = 1: 128 positions per tile
    ("bf16", 128, 1, [200], [260]),
    # fp32 chunk (CUDA-core path) with splits
    ("f32", 128, 2, [100, 1], [700, 300]),
    # fewer tensor-core units than SMs: each query tile's KV is split into
    # pieces whose partial states the last piece merges
    ("bf16", 128, 4, [20, 1], [9000, 3000]),
    ("bf16", 64, 8, [40, 1], [6000, 17]),
    # G = 1, 128 positions per tile: a piece boundary (key 4096) falls inside
    # the first query tile, so its early rows see no key in the last piece
    ("bf16", 128, 1, [150], [4150]),
    # units of 157, 16 and 6 KV tiles, fewer than SMs: the plan takes the
    # smallest piece size that fits one round, cutting them unevenly
    ("bf16", 128, 4, [16, 16, 48], [20000, 2000, 700]),
]


@pytest.mark.parametrize("case", range(len(PREFILL_SHAPES)))
def test_prefill_shapes(case):
    dtype, D, G, q_lens, seq_lens = PREFILL_SHAPES[case]
    spec = W.custom_spec(f"prefill-{case}", dtype, 2 * G, 2, D, q_lens, seq_lens, seed=200 + case)
    _full_parity(W.make_step(spec))


def _rising_logits(step, slope_log2: float, qmag: float = 8.0, seed: int = 5):
    """Make every row's logits grow along the key positions: keys of position
    p are u * c * p and query rows u * qmag for one unit vector u, so the base-2
    logit of key p is slope_log2 * p.  The running maximum then moves by more
    than the kernels' lazy-rescale threshold within 64 keys, which drives the
    rescale paths."""
    import math
    spec = step.spec
    D = spec.head_size
    u = torch.randn(D, generator=torch.Generator().manual_seed(seed))
    u = u / u.norm()
    c = slope_log2 / (step.scale * math.log2(math.e) * qmag)
    dt = step.q.dtype
    step.q[:] = (u * qmag).to(dt)
    bt = step.block_tables.numpy()
    qsl = step.query_start_loc.numpy()
    flat_k = step.k_cache.view(-1, spec.num_kv_heads, D)
    for r in range(spec.num_seqs):
        S, L = int(spec.seq_lens[r]), int(spec.q_lens[r])
        for pos in range(S):
            key = (u * (c * pos)).to(dt)
            if pos < S - L:
                slot = int(bt[r, pos // 16]) * 16 + pos % 16
                flat_k[slot] = key
            else:
                step.k[int(qsl[r]) + pos - (S - L)] = key
    return step


def test_rescale_paths_rising_logits():
    """Logits rising by 0.2 (base 2) per key: the prefill kernel's O rescale and
    its second-half P fix-up, and the decode kernel's running-maximum updates,
    all run; the result still matches the oracle."""
    spec = W.custom_spec("rising", "bf16", 8, 2, 128, [300, 1], [1200, 700], seed=41)
    _full_parity(_rising_logits(W.make_step(spec), slope_log2=0.2))
