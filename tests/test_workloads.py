"""The seeded input generator: shapes, determinism and valid block tables (no GPU)."""
import numpy as np

from paged_kv_attention_18_gb300 import workloads as W


def _check_tables(wl):
    for st in wl.steps:
        assert st.block_tables.dtype == np.int32
        for b in range(st.B):
            L = int(st.seq_lens[b])
            nblk = -(-L // 16)
            row = st.block_tables[b]
            assert ((row[:nblk] >= 0) & (row[:nblk] < wl.num_blocks)).all()
            # entries past the context are -1 padding or blocks held for later tokens
            assert (row[nblk:] >= -1).all()
        n = np.diff(st.query_start_loc)
        assert (n <= st.seq_lens).all()
        assert st.q.shape == (st.T, wl.H_q, wl.D) and st.k.shape == (st.T, wl.H_kv, wl.D)


def test_tiny_decode():
    wl = W.tiny_decode()
    assert (wl.H_q, wl.H_kv, wl.D, wl.dtype, wl.num_blocks) == (4, 2, 64, "f16", 64)
    st = wl.steps[0]
    assert st.B == 4 and st.T == 4 and ((st.seq_lens >= 1) & (st.seq_lens <= 100)).all()
    _check_tables(wl)
    again = W.tiny_decode()
    assert np.array_equal(again.k_pool, wl.k_pool) and np.array_equal(again.steps[0].q, st.q)


def test_mixed_shapes():
    wl = W.qwen05b_mixed()
    st = wl.steps[0]
    assert st.T == 520 and st.B == 10 and wl.num_blocks == 2048
    assert st.seq_lens[8:].tolist() == [256, 768]
    assert np.diff(st.query_start_loc).tolist() == [1] * 8 + [256, 256]
    _check_tables(wl)


def test_private_blocks_distinct_and_prefix_shared():
    wl = W.prefix_chunked_prefill(n_prefill=6, prefix_tokens=64, suffix_lo=20, suffix_hi=60,
                                  n_decode=3, dec_lo=16, dec_hi=40, budget=64)
    assert len(wl.steps) > 1
    _check_tables(wl)
    seen = {}
    for st in wl.steps:
        for b in range(st.B):
            seen[int(st.seq_ids[b])] = st.block_tables[b]
    prefix = [tuple(seen[i][:4]) for i in range(6)]
    assert len(set(prefix)) == 1
    blocks = [blk for i, row in seen.items() for blk in row[(4 if i < 6 else 0):] if blk >= 0]
    assert len(blocks) == len(set(blocks))
    for st in wl.steps:  # every step within the budget, decodes first
        assert st.T <= 64
        assert np.diff(st.query_start_loc)[:3].tolist() == [1, 1, 1]


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38], dtype=np.float32)
    bits = W.round_to_bits(x, "bf16")
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert back.tolist()[:4] == [1.0, 1.0, 1.015625, -2.5]  # ties go to even


def test_verify_shapes_small():
    wl = W.spec_verify_long(n_seq=4, lo=16, hi=64, n_long=1, long_len=200)
    st = wl.steps[0]
    assert st.B == 5 and st.T == 25 and st.seq_lens[-1] == 200
    _check_tables(wl)
