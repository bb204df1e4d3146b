"""Oracle pins for attention over per-row key lists (the index-list gather).

TensorSharp "高级功能", the DeepSeek V4 executor item: decode attention reads a compact
[ring | top-512] set of keys through an index-gather instead of the whole context.
Pinned against the (separately pinned) paged attention oracle: a list naming every key
in order is the dense attention, bit for bit; list order only changes rounding; a
one-key list returns that key's V row; a key listed twice weighs twice.
"""
import numpy as np
import pytest

from paged_kv_attention_forward_gb300 import workloads as wl


def _batch(seed=0, lens=(37, 100, 203), Hq=8, Hkv=2, D=64, B=16, sinks=False):
    lens = np.array(lens)
    return wl.build_batch(seed, name="t", lens=lens, n_new=np.zeros(len(lens), np.int64),
                          q_rows=np.ones(len(lens), np.int64), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                          block_size=B, causal=False, with_sinks=sinks)


def _lists(rows):
    width = max(len(r) for r in rows)
    idx = np.full((len(rows), width), -1, np.int32)
    for i, r in enumerate(rows):
        idx[i, :len(r)] = r
    return idx, np.array([len(r) for r in rows], np.int32)


@pytest.mark.parametrize("sinks", [False, True])
def test_full_list_in_order_is_dense_attention(oracle_mod, sinks):
    b = _batch(sinks=sinks)
    idx, cnt = _lists([np.arange(L) for L in b.context_lens])
    dense = oracle_mod.paged_attention(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables,
                                       b.context_lens, sinks=b.sinks)
    got = oracle_mod.paged_attention_sparse(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables,
                                            b.context_lens, idx, cnt, sinks=b.sinks)
    assert np.array_equal(got, dense)


def test_list_order_only_changes_rounding(oracle_mod):
    b = _batch(1)
    rng = np.random.default_rng(1)
    rows = [rng.choice(L, size=min(L, 30), replace=False) for L in b.context_lens]
    idx, cnt = _lists(rows)
    idx2, _ = _lists([r[::-1] for r in rows])
    a = oracle_mod.paged_attention_sparse(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables,
                                          b.context_lens, idx, cnt)
    c = oracle_mod.paged_attention_sparse(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables,
                                          b.context_lens, idx2, cnt)
    assert np.allclose(a, c, rtol=0, atol=1e-12)


def test_one_key_and_repeated_keys(oracle_mod):
    b = _batch(2)
    kp, vp = b.k_pool[0], b.v_pool[0]
    t_a, t_b = 5, 20
    s = 1                                                   # row 1 = sequence 1
    idx, cnt = _lists([[0], [t_a], [0]])
    one = oracle_mod.paged_attention_sparse(kp, vp, b.q[0], b.q_starts, b.block_tables, b.context_lens, idx, cnt)
    def row_of(t, g):
        blk = b.block_tables[s, t // 16]
        return wl.bf16_bits_to_f32(vp[blk, g, t % 16]).astype(np.float64)
    for h in range(8):
        assert np.array_equal(one[1, h], row_of(t_a, h // 4))   # softmax over one key
    # [a, a, b]: a weighs twice as much as in [a, b]
    idx3, cnt3 = _lists([[0], [t_a, t_a, t_b], [0]])
    got = oracle_mod.paged_attention_sparse(kp, vp, b.q[0], b.q_starts, b.block_tables, b.context_lens, idx3, cnt3)
    for h in range(8):
        g = h // 4
        blk_a, blk_b = b.block_tables[s, t_a // 16], b.block_tables[s, t_b // 16]
        q = wl.bf16_bits_to_f32(b.q[0][1, h]).astype(np.float64)
        ka = wl.bf16_bits_to_f32(kp[blk_a, g, t_a % 16]).astype(np.float64)
        kb = wl.bf16_bits_to_f32(kp[blk_b, g, t_b % 16]).astype(np.float64)
        xa, xb = q @ ka / 8.0, q @ kb / 8.0
        m = max(xa, xb)
        wa, wb = 2 * np.exp(xa - m), np.exp(xb - m)
        ref = (wa * row_of(t_a, g) + wb * row_of(t_b, g)) / (wa + wb)
        assert np.allclose(got[1, h], ref, rtol=1e-12, atol=1e-12)


def test_empty_list_and_bad_positions(oracle_mod):
    b = _batch(3)
    idx, cnt = _lists([[0], [1], [2]])
    cnt[0] = 0
    out = oracle_mod.paged_attention_sparse(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables,
                                            b.context_lens, idx, cnt)
    assert not out[0].any()
    idx[1, 0] = int(b.context_lens[1])                      # one past the context
    with pytest.raises(ValueError):
        oracle_mod.paged_attention_sparse(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables,
                                          b.context_lens, idx, cnt)


def test_key_list_generator():
    b = wl.make_workload("tiny_decode")
    wl.add_key_lists(b, 5, ring=16, top=40, sets=2)
    for k in range(2):
        for r in range(b.total_q_rows):
            n = b.key_counts[k, r]
            lst = b.key_idx[k, r, :n]
            L = int(b.context_lens[r])
            assert len(set(lst.tolist())) == n and lst.min() >= 0 and lst.max() < L
            assert np.array_equal(lst[:min(16, L)], np.arange(L - min(16, L), L))
            assert np.all(b.key_idx[k, r, n:] == -1)
