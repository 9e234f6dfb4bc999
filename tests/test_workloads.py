"""The seeded workloads have the structure the configurations describe."""
import math

import numpy as np
import pytest

import oracle
from paged_kv_attention_04_gb300 import workloads as W


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_metadata_consistent(name):
    spec = W.CONFIGS[name]()
    m = W.make_meta(spec)
    oracle.validate_step(m.block_tables, spec.seq_lens, m.query_start_loc, m.num_blocks,
                         m.slot_mapping)
    # every new token's slot follows its request's table
    qsl = m.query_start_loc
    for r in range(spec.num_seqs):
        S, L = int(spec.seq_lens[r]), int(spec.q_lens[r])
        want = [oracle.slot_of(m.block_tables[r], p) for p in range(S - L, S)]
        assert list(m.slot_mapping[qsl[r]:qsl[r + 1]]) == want
        nb = oracle.blocks_needed(S)
        assert np.all(m.block_tables[r, nb:] == -1)


def test_config_shapes():
    s1 = W.spec_tiny_decode_f32()
    assert list(s1.seq_lens) == [1, 17, 33, 64] and s1.num_blocks == 32
    m1 = W.make_meta(s1)
    assert m1.unique_blocks == 1 + 2 + 3 + 4
    # non-contiguous tables
    assert any(np.any(np.diff(row[row >= 0]) != 1) for row in m1.block_tables)

    s2 = W.spec_tinyllama_decode()
    assert s2.num_seqs == 64 and s2.seq_lens.min() >= 128 and s2.seq_lens.max() <= 2048
    m2 = W.make_meta(s2)
    assert m2.num_blocks == math.ceil(1.2 * m2.unique_blocks)

    s3 = W.spec_llama3_8b_decode()
    assert s3.num_seqs == 256 and s3.seq_lens.max() <= 8192 and s3.seq_lens.min() >= 1
    assert 700 < np.median(s3.seq_lens) < 1400

    s4 = W.spec_mixed_step()
    m4 = W.make_meta(s4)
    assert s4.num_tokens == 1216
    assert list(m4.query_start_loc[190:]) == [190, 191, 192, 704, 1216]
    assert list(s4.seq_lens[192:]) == [512, 2048]
    dec = s4.seq_lens[:192]
    assert dec.min() >= 256 and dec.max() <= 4096
    # 96 sharing requests map their first min(64, (S-1)//16) blocks to one set
    shared_rows = np.nonzero(s4.sharing)[0]
    assert len(shared_rows) == 96
    common = m4.block_tables[shared_rows[0], :1]
    for r in shared_rows:
        k = min(64, (int(s4.seq_lens[r]) - 1) // 16)
        assert np.all(m4.block_tables[r, :1] == common)
        ids = m4.block_tables[r, :k]
        assert len(set(ids.tolist())) == k
    others = [r for r in range(194) if not s4.sharing[r]]
    used_by_others = set(m4.block_tables[others].ravel().tolist()) - {-1}
    assert not (set(m4.block_tables[shared_rows[0], :1].tolist()) & used_by_others)

    s5 = W.spec_long_context_decode()
    assert s5.num_blocks == 137329 and s5.num_seqs == 16
    assert s5.seq_lens.min() >= 32768 and s5.seq_lens.max() <= 131072
    m5 = W.make_meta(s5)
    assert m5.unique_blocks <= 137329

    s6 = W.spec_long_prefill_chunk()
    m6 = W.make_meta(s6)
    assert list(s6.q_lens) == [2048] and list(s6.seq_lens) == [8192]
    assert list(m6.query_start_loc) == [0, 2048] and m6.unique_blocks == 512


def test_tensors_and_nan_pool():
    spec = W.spec_tiny_decode_f32()
    st = W.make_step(spec)
    m = W.make_meta(spec)
    assert st.q.shape == (4, 4, 64) and st.k.shape == (4, 2, 64)
    assert st.k_cache.shape == (32, 16, 2, 64)
    flat = st.k_cache.reshape(-1, 2, 64)
    hist = np.nonzero(m.hist_mask)[0]
    assert flat[hist].isfinite().all()
    nothist = np.nonzero(~m.hist_mask)[0]
    assert flat[nothist].isnan().all()
    # the slots this step writes hold NaN before the write
    assert flat[st.slot_mapping].isnan().all()
    # seeded: the same spec gives the same bits
    st2 = W.make_step(W.spec_tiny_decode_f32())
    assert st.q.equal(st2.q) and st.k_cache.nan_to_num().equal(st2.k_cache.nan_to_num())


def test_bf16_tensors_round_from_f32():
    spec = W.custom_spec("small", "bf16", 4, 2, 64, [1, 3], [20, 40])
    st = W.make_step(spec)
    assert st.q.dtype.is_floating_point and str(st.q.dtype) == "torch.bfloat16"
    bits = W.to_numpy_bits(st.q)
    assert bits.dtype == np.uint16 and bits.shape == (4, 4, 64)
