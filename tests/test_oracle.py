"""Pins for the fp64 oracle: checks that do not go through the oracle's own
formulas.  Each would fail on a plausible slip in the oracle (a dropped scale,
a wrong sign, a wrong kv-head mapping, an off-by-one in the causal limit, a
transposed block/row index)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_04_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def _paged_from_contiguous(Kc, Vc, block_size, num_blocks, rng):
    """Scatter contiguous per-request KV [S][Hkv][D] into a fresh paged pool
    through a random permutation of physical blocks.  Written here, apart
    from the oracle, with a flat slot view: slot = block * bs + row."""
    Hkv, D = Kc[0].shape[1:]
    kc = np.full((num_blocks, block_size, Hkv, D), np.nan)
    vc = np.full_like(kc, np.nan)
    perm = rng.permutation(num_blocks)
    tables, cur = [], 0
    maxnb = max(-(-len(k) // block_size) for k in Kc)
    for K, V in zip(Kc, Vc):
        nb = -(-len(K) // block_size)
        row = np.full(maxnb, -1, np.int64)
        row[:nb] = perm[cur:cur + nb]
        cur += nb
        slots = row[np.arange(len(K)) // block_size] * block_size + np.arange(len(K)) % block_size
        kc.reshape(-1, Hkv, D)[slots] = K
        vc.reshape(-1, Hkv, D)[slots] = V
        tables.append(row)
    return kc, vc, np.stack(tables)


def _random_step(rng, q_lens, seq_lens, Hq, Hkv, D, block_size=16, extra_blocks=5):
    Kc = [rng.standard_normal((s, Hkv, D)) for s in seq_lens]
    Vc = [rng.standard_normal((s, Hkv, D)) for s in seq_lens]
    nb = sum(-(-s // block_size) for s in seq_lens) + extra_blocks
    kc, vc, bt = _paged_from_contiguous(Kc, Vc, block_size, nb, rng)
    T = int(sum(q_lens))
    q = rng.standard_normal((T, Hq, D))
    qsl = np.concatenate([[0], np.cumsum(q_lens)])
    return q, kc, vc, bt, np.array(seq_lens), qsl, Kc, Vc


# ---------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_block_count_examples():
    rows = _rows("block_count.txt")
    assert rows, "fixture empty"
    for n, bs, want in rows:
        assert oracle.blocks_needed(int(n), int(bs)) == int(want)


def test_block_count_against_brute_fill():
    # fill blocks one token at a time; count the blocks opened
    for bs in (1, 4, 16):
        for n in range(0, 70):
            opened, room = 0, 0
            for _ in range(n):
                if room == 0:
                    opened, room = opened + 1, bs
                room -= 1
            assert oracle.blocks_needed(n, bs) == opened


def test_block_table_req2_slots():
    rows = _rows("block_table_req2.txt")
    table = [2, 5, 8]
    for pos, want in rows:
        assert oracle.slot_of(table, int(pos), 16) == int(want)


def test_block_bytes_matches_allocated_block():
    # bytes one physical block of the generated K and V pools occupies
    for name in ("tiny_decode_f32", "tinyllama_decode"):
        spec = W.CONFIGS[name]()
        spec.seq_lens = spec.seq_lens[:2]
        spec.q_lens = spec.q_lens[:2]
        st = W.make_step(spec)
        got = st.k_cache[0].numel() * st.k_cache.element_size() * 2
        e = 4 if spec.dtype == "f32" else 2
        assert oracle.block_bytes(spec.num_kv_heads, spec.head_size, e) == got
    # the Llama-3-8B block is the 64 KiB that sizes the long-context pool
    assert oracle.block_bytes(8, 128, 2) == 65536 == int(9e9) // 137329


def test_shared_prefix_block_reads_same_kv():
    rows = _rows("shared_prefix.txt")
    tab = {}
    for req, lb, pb in rows:
        tab.setdefault(req, {})[int(lb)] = int(pb)
    bt = np.full((2, 2), -1, np.int64)
    bt[0, 0], bt[0, 1] = tab["A"][0], tab["A"][1]
    bt[1, 0] = tab["B"][0]
    rng = np.random.default_rng(7)
    Hkv, D = 1, 8
    kc = rng.standard_normal((64, 16, Hkv, D))
    vc = rng.standard_normal((64, 16, Hkv, D))
    # A has 20 tokens (two blocks), B has 16: B's whole context is A's block #42
    seq = np.array([20, 16])
    qv = rng.standard_normal((1, 1, D))
    # A runs a 5-token chunk (positions 15..19): its first row sees exactly
    # block #42, like B's decode row at position 15
    qA = np.repeat(qv, 5, axis=0)
    q = np.concatenate([qA, qv])
    qsl = np.array([0, 5, 6])
    out = oracle.paged_attention(q, kc, vc, bt, seq, qsl, 0.5, num_kv_heads=Hkv)
    np.testing.assert_array_equal(out[0], out[5])
    assert not np.array_equal(out[1], out[5])


def test_scheduler_step_layout():
    f = {r[0]: [int(x) for x in r[1:]] for r in _rows("scheduler_step.txt")}
    q_lens = f["q_lens"]
    assert sum(q_lens) == f["budget"][0] - f["left"][0]
    assert f["waiting_prompt"][0] > f["left"][0]
    spec = W.custom_spec("sched", "f32", 2, 1, 8, q_lens, [5, 9, 3, 6])
    st = W.make_step(spec)
    assert st.query_start_loc.tolist() == f["query_start_loc"]
    oracle.validate_step(st.block_tables.numpy(), st.seq_lens.numpy(),
                         st.query_start_loc.numpy(), st.num_blocks, st.slot_mapping.numpy())


# ---------------------------------------------------------------------------
# Element widening
# ---------------------------------------------------------------------------

def test_widen_bf16_known_bits():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x0001, 0x3E80], np.uint16)
    got = oracle.widen(bits)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 0.0
    assert math.copysign(1.0, got[3]) == -1.0 and got[4] == math.inf
    assert got[5] == 2.0 ** -133 and got[6] == 0.25


def test_widen_bf16_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(4096, generator=g).mul(100).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.widen(bits), x.to(torch.float64).numpy())


# ---------------------------------------------------------------------------
# Slot write
# ---------------------------------------------------------------------------

def test_cache_write_flat_view_and_untouched():
    rng = np.random.default_rng(1)
    NB, bs, Hkv, D, T = 6, 16, 2, 8, 11
    kc0 = rng.integers(0, 2 ** 16, (NB, bs, Hkv, D)).astype(np.uint16)
    vc0 = rng.integers(0, 2 ** 16, (NB, bs, Hkv, D)).astype(np.uint16)
    k = rng.integers(0, 2 ** 16, (T, Hkv, D)).astype(np.uint16)
    v = rng.integers(0, 2 ** 16, (T, Hkv, D)).astype(np.uint16)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    slots[3] = -1
    kc, vc = oracle.cache_write(k, v, slots, kc0, vc0)
    ek, ev = kc0.copy().reshape(-1, Hkv, D), vc0.copy().reshape(-1, Hkv, D)
    live = slots >= 0
    ek[slots[live]] = k[live]
    ev[slots[live]] = v[live]
    np.testing.assert_array_equal(kc.reshape(-1, Hkv, D), ek)
    np.testing.assert_array_equal(vc.reshape(-1, Hkv, D), ev)
    # inputs not modified
    assert not np.shares_memory(kc, kc0)


# ---------------------------------------------------------------------------
# Attention: closed forms
# ---------------------------------------------------------------------------

def test_seq_len_one_returns_v0():
    rng = np.random.default_rng(2)
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, [1, 1], [1, 1], 4, 2, 16)
    out = oracle.paged_attention(q, kc, vc, bt, S, qsl, 0.25, num_kv_heads=2)
    for r in range(2):
        for h in range(4):
            np.testing.assert_array_equal(out[r, h], Vc[r][0, h // 2])


def test_zero_query_gives_mean_of_visible_v():
    rng = np.random.default_rng(3)
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, [3, 1], [21, 40], 2, 1, 8)
    q[:] = 0.0
    out = oracle.paged_attention(q, kc, vc, bt, S, qsl, 1.0, num_kv_heads=1)
    for j in range(3):
        pos = 21 - 3 + j
        np.testing.assert_allclose(out[j, 0], Vc[0][:pos + 1, 0].mean(0), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out[3, 1], Vc[1][:, 0].mean(0), rtol=1e-13, atol=1e-13)


def test_constant_v_is_returned():
    rng = np.random.default_rng(4)
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, [5], [37], 4, 4, 8)
    vc[:] = 0.75
    out = oracle.paged_attention(q * 9.0, kc, vc, bt, S, qsl, 0.3, num_kv_heads=4)
    np.testing.assert_allclose(out, 0.75, rtol=1e-14)


def test_one_dominant_key_selects_its_value():
    # scale * q.k huge at one visible position p*: output -> V[p*]
    rng = np.random.default_rng(5)
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, [1], [33], 1, 1, 4)
    q[0, 0] = np.array([1.0, 0, 0, 0])
    pstar = 20
    slot = bt[0, pstar // 16] * 16 + pstar % 16
    kc.reshape(-1, 1, 4)[slot, 0] = [400.0, 0, 0, 0]
    out = oracle.paged_attention(q, kc, vc, bt, S, qsl, 1.0, num_kv_heads=1)
    np.testing.assert_allclose(out[0, 0], Vc[0][pstar, 0], atol=1e-12)


# ---------------------------------------------------------------------------
# Attention: against a library routine and a brute-force loop
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("Hq,Hkv,D", [(4, 2, 16), (8, 1, 8), (6, 3, 32), (2, 2, 64)])
def test_matches_torch_sdpa_on_contiguous_kv(Hq, Hkv, D):
    rng = np.random.default_rng(Hq * 100 + D)
    q_lens = [1, 7, 1, 16, 3]
    seq_lens = [1, 30, 17, 16, 50]
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, q_lens, seq_lens, Hq, Hkv, D)
    scale = 1.0 / math.sqrt(D) * 1.7
    out = oracle.paged_attention(q, kc, vc, bt, S, qsl, scale, num_kv_heads=Hkv)
    G = Hq // Hkv
    for r, (L, s) in enumerate(zip(q_lens, seq_lens)):
        Q = torch.from_numpy(q[qsl[r]:qsl[r + 1]]).permute(1, 0, 2)           # [Hq][L][D]
        K = torch.from_numpy(Kc[r]).permute(1, 0, 2).repeat_interleave(G, 0)  # [Hq][S][D]
        V = torch.from_numpy(Vc[r]).permute(1, 0, 2).repeat_interleave(G, 0)
        # bottom-right aligned causal mask: row j sees keys 0 .. s - L + j
        mask = torch.arange(s)[None, :] <= (s - L + torch.arange(L))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(out[qsl[r]:qsl[r + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_matches_pure_python_brute_force():
    rng = np.random.default_rng(11)
    q_lens, seq_lens = [2, 1, 4], [3, 18, 20]
    Hq, Hkv, D = 4, 2, 4
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, q_lens, seq_lens, Hq, Hkv, D)
    scale = 0.37
    out = oracle.paged_attention(q, kc, vc, bt, S, qsl, scale, num_kv_heads=Hkv)
    for r in range(3):
        L, s = q_lens[r], seq_lens[r]
        for j in range(L):
            t = qsl[r] + j
            for h in range(Hq):
                g = h * Hkv // Hq
                xs = []
                for p in range(s - L + j + 1):
                    acc = 0.0
                    for d in range(D):
                        acc += q[t, h, d] * Kc[r][p, g, d]
                    xs.append(scale * acc)
                mx = max(xs)
                ws = [math.exp(x - mx) for x in xs]
                tot = sum(ws)
                for d in range(D):
                    o = sum(w * Vc[r][p, g, d] for p, w in enumerate(ws)) / tot
                    assert abs(out[t, h, d] - o) <= 1e-12 * (1 + abs(o))


def test_rows_api_matches_full():
    rng = np.random.default_rng(12)
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, [1, 5, 1], [9, 40, 70], 8, 2, 16)
    full = oracle.paged_attention(q, kc, vc, bt, S, qsl, 0.25, num_kv_heads=2)
    rows = [(0, 3), (1, 0), (3, 7), (5, 5), (6, 1)]
    part = oracle.paged_attention_rows(q, kc, vc, bt, S, qsl, 0.25, 2, rows)
    for i, (t, h) in enumerate(rows):
        np.testing.assert_allclose(part[i], full[t, h], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# Attention: invariances the pages fix
# ---------------------------------------------------------------------------

def test_physical_block_permutation_invariance():
    rng = np.random.default_rng(13)
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, [1, 3, 1], [17, 33, 64], 4, 2, 16)
    out = oracle.paged_attention(q, kc, vc, bt, S, qsl, 0.25, num_kv_heads=2)
    NB = kc.shape[0]
    perm = rng.permutation(NB)            # physical block b moves to perm[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    out2 = oracle.paged_attention(q, kc2, vc2, bt2, S, qsl, 0.25, num_kv_heads=2)
    np.testing.assert_array_equal(out, out2)


def test_batch_invariance():
    rng = np.random.default_rng(14)
    q_lens, seq_lens = [1, 4, 1], [20, 25, 5]
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, q_lens, seq_lens, 2, 1, 8)
    out = oracle.paged_attention(q, kc, vc, bt, S, qsl, 0.4, num_kv_heads=1)
    for r in range(3):
        alone = oracle.paged_attention(q[qsl[r]:qsl[r + 1]], kc, vc, bt[r:r + 1], S[r:r + 1],
                                       np.array([0, q_lens[r]]), 0.4, num_kv_heads=1)
        np.testing.assert_array_equal(alone, out[qsl[r]:qsl[r + 1]])


def test_chunked_prefill_equals_unchunked():
    # the page's example: chunks of 8 tokens, an 18-token prompt x-y-z
    rng = np.random.default_rng(15)
    Hq, Hkv, D, n = 4, 2, 8, 18
    Kp = rng.standard_normal((n, Hkv, D))
    Vp = rng.standard_normal((n, Hkv, D))
    Qp = rng.standard_normal((n, Hq, D))
    NB = 4
    bt = np.array([[3, 1]])
    empty = np.full((NB, 16, Hkv, D), np.nan)
    # unchunked: write all 18, attend with q_len 18
    slots = np.array([oracle.slot_of(bt[0], p) for p in range(n)])
    kc, vc = oracle.cache_write(Kp, Vp, slots, empty, empty)
    full = oracle.paged_attention(Qp, kc, vc, bt, np.array([n]), np.array([0, n]), 0.3, Hkv)
    # chunked: 8, 8, 2 tokens, each chunk written then attended
    kc, vc = empty.copy(), empty.copy()
    done, outs = 0, []
    for c in (8, 8, 2):
        kc, vc = oracle.cache_write(Kp[done:done + c], Vp[done:done + c], slots[done:done + c], kc, vc)
        outs.append(oracle.paged_attention(Qp[done:done + c], kc, vc, bt, np.array([done + c]),
                                           np.array([0, c]), 0.3, Hkv))
        done += c
    np.testing.assert_allclose(np.concatenate(outs), full, rtol=1e-14, atol=1e-14)


def test_decode_equals_last_prefill_row():
    rng = np.random.default_rng(16)
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, [9], [30], 4, 2, 16)
    pre = oracle.paged_attention(q, kc, vc, bt, S, qsl, 0.25, 2)
    dec = oracle.paged_attention(q[-1:], kc, vc, bt, S, np.array([0, 1]), 0.25, 2)
    np.testing.assert_array_equal(pre[-1], dec[0])


def test_unwritten_slots_are_never_read():
    # NaN in a request's last block beyond seq_len, and in unused blocks
    rng = np.random.default_rng(17)
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, [1, 2], [17, 31], 2, 2, 8)
    out = oracle.paged_attention(q, kc, vc, bt, S, qsl, 0.25, 2)
    assert np.isfinite(out).all()


# ---------------------------------------------------------------------------
# Validation catches malformed steps (the mistakes are planted in inputs)
# ---------------------------------------------------------------------------

def test_validate_rejects_bad_steps():
    bt = np.array([[0, 1], [2, -1]])
    S = np.array([20, 5])
    ok_qsl = np.array([0, 1, 3])
    oracle.validate_step(bt, S, ok_qsl, 3, np.array([19, 33, 34]))
    with pytest.raises(ValueError):
        oracle.validate_step(bt, S, np.array([0, 2, 1]), 3)
    with pytest.raises(ValueError):
        oracle.validate_step(bt, np.array([20, 1]), ok_qsl, 3)          # q_len 2 > seq_len 1
    with pytest.raises(ValueError):
        oracle.validate_step(bt, S, ok_qsl, 2)                          # block 2 outside 2-block pool
    with pytest.raises(ValueError):
        oracle.validate_step(bt, S, ok_qsl, 3, np.array([19, 33, 33]))  # duplicate slot
    with pytest.raises(ValueError):
        oracle.validate_step(bt, S, ok_qsl, 3, np.array([19, 33, 48]))  # slot outside pool


def test_planted_mistakes_are_caught():
    """Each plausible slip, planted in a copy of the oracle's formula here on
    the CPU, disagrees with the library reference (torch SDPA)."""
    rng = np.random.default_rng(18)
    q_lens, seq_lens, Hq, Hkv, D = [3], [21], 4, 2, 8
    q, kc, vc, bt, S, qsl, Kc, Vc = _random_step(rng, q_lens, seq_lens, Hq, Hkv, D)
    scale = 0.3
    G = Hq // Hkv
    Q = torch.from_numpy(q).permute(1, 0, 2)
    K = torch.from_numpy(Kc[0]).permute(1, 0, 2).repeat_interleave(G, 0)
    V = torch.from_numpy(Vc[0]).permute(1, 0, 2).repeat_interleave(G, 0)
    mask = torch.arange(21)[None, :] <= (21 - 3 + torch.arange(3))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                           scale=scale).permute(1, 0, 2).numpy()

    def variant(scale_on=True, head_map=lambda h: h // G, causal_off=0):
        out = np.empty_like(ref)
        for j in range(3):
            pos = 21 - 3 + j + causal_off
            for h in range(Hq):
                g = head_map(h)
                x = (scale if scale_on else 1.0) * (Kc[0][:pos + 1, g] @ q[j, h])
                w = np.exp(x - x.max())
                out[j, h] = w @ Vc[0][:pos + 1, g] / w.sum()
        return out

    np.testing.assert_allclose(variant(), ref, rtol=1e-12, atol=1e-12)
    for bad in (variant(scale_on=False), variant(head_map=lambda h: h % Hkv),
                variant(causal_off=-1)):
        assert not np.allclose(bad, ref, rtol=1e-6, atol=1e-6)
