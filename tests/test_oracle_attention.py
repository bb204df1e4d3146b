"""Pins for the float64 attention oracle (no GPU).

Each test checks the oracle against something other than itself: torch's float64
scaled-dot-product attention on contiguous K/V, closed forms, invariances the
definition implies, and a hand-worked fixture.  Definition followed: TensorSharp
"高级功能", sections "连续批处理与分页 KV 缓存" and "原生分页注意力" (paged K/V gather,
optional per-head sinks); the causal verify window follows the TensorFold article,
section "先记住一条铁律" (every verify row uses the serial step's attention bounds).
"""
import math
import os

import numpy as np
import pytest
import torch

from paged_kv_attention_forward_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return wl.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _pool_from_contiguous(oracle_mod, rng, seqs_k, seqs_v, B, nb_extra=3):
    """Write contiguous per-sequence K/V into a fresh pool through the oracle's append,
    one token at a time, with physical blocks drawn from a random permutation."""
    S = len(seqs_k)
    H, D = seqs_k[0].shape[1], seqs_k[0].shape[2]
    lens = [k.shape[0] for k in seqs_k]
    nblk = [(L + B - 1) // B for L in lens]
    num_blocks = sum(nblk) + nb_extra
    perm = rng.permutation(num_blocks).astype(np.int32)
    maxb = max(1, max(nblk))
    tables = np.full((S, maxb), -1, np.int32)
    c = 0
    for s in range(S):
        tables[s, :nblk[s]] = perm[c:c + nblk[s]]
        c += nblk[s]
    kp = _bf16(rng.standard_normal((num_blocks, H, B, D)))
    vp = _bf16(rng.standard_normal((num_blocks, H, B, D)))
    for t in range(max(lens)):
        ss = [s for s in range(S) if t < lens[s]]
        old = np.array([t if s in ss else lens[s] for s in range(S)], np.int32)
        cnt = np.array([1 if s in ss else 0 for s in range(S)])
        ns = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        kn = np.stack([seqs_k[s][t] for s in ss]) if ss else np.zeros((0, H, D), np.uint16)
        vn = np.stack([seqs_v[s][t] for s in ss]) if ss else np.zeros((0, H, D), np.uint16)
        oracle_mod.paged_kv_append(kp, vp, tables, old, ns, kn, vn)
    return kp, vp, tables, np.array(lens, np.int32)


def _sdpa_reference(q_rows, K, V, G, causal_rows=None, scale=None, head_map=None):
    """torch float64 SDPA on one sequence's contiguous K/V.  q_rows [W, Hq, D] f64,
    K/V [L, Hkv, D] f64.  head_map: q head -> kv head (None: contiguous groups)."""
    W, Hq, D = q_rows.shape
    L = K.shape[0]
    if head_map is None:
        head_map = [h // G for h in range(Hq)]
    Kx = torch.from_numpy(K[:, head_map, :]).permute(1, 0, 2)  # [Hq, L, D]
    Vx = torch.from_numpy(V[:, head_map, :]).permute(1, 0, 2)
    Q = torch.from_numpy(q_rows).permute(1, 0, 2)             # [Hq, W, D]
    mask = None
    if causal_rows is not None:
        t = torch.arange(L)[None, :]
        lim = torch.tensor(causal_rows)[:, None]
        mask = t < lim                                          # [W, L]
    out = torch.nn.functional.scaled_dot_product_attention(
        Q[None], Kx[None], Vx[None], attn_mask=mask, scale=scale)
    return out[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(oracle_mod, causal):
    rng = np.random.default_rng(1234)
    B, H, G, D = 4, 2, 3, 16
    lens = [1, 7, 17, 50]
    W = [1, 2, 1, 5]
    seqs_k = [_bf16(rng.standard_normal((L, H, D))) for L in lens]
    seqs_v = [_bf16(rng.standard_normal((L, H, D))) for L in lens]
    kp, vp, tables, cl = _pool_from_contiguous(oracle_mod, rng, seqs_k, seqs_v, B)
    q_starts = np.concatenate([[0], np.cumsum(W)]).astype(np.int32)
    q = _bf16(rng.standard_normal((q_starts[-1], H * G, D)))
    out = oracle_mod.paged_attention(kp, vp, q, q_starts, tables, cl, causal=causal)
    for s, L in enumerate(lens):
        rows = slice(q_starts[s], q_starts[s + 1])
        lim = [L - W[s] + w + 1 for w in range(W[s])] if causal else None
        ref = _sdpa_reference(_f64(q[rows]), _f64(seqs_k[s]), _f64(seqs_v[s]), G, lim)
        np.testing.assert_allclose(out[rows], ref, rtol=0, atol=1e-12)


def test_explicit_head_map_matches_sdpa(oracle_mod):
    rng = np.random.default_rng(7)
    B, H, G, D = 4, 3, 2, 8
    hmap = np.array([2, 0, 1, 0, 2, 1], np.int32)   # each kv head serves G=2 q heads
    seqs_k = [_bf16(rng.standard_normal((L, H, D))) for L in (9, 4)]
    seqs_v = [_bf16(rng.standard_normal((L, H, D))) for L in (9, 4)]
    kp, vp, tables, cl = _pool_from_contiguous(oracle_mod, rng, seqs_k, seqs_v, B)
    q_starts = np.array([0, 1, 2], np.int32)
    q = _bf16(rng.standard_normal((2, H * G, D)))
    out = oracle_mod.paged_attention(kp, vp, q, q_starts, tables, cl, kv_head_of_q_head=hmap)
    for s in range(2):
        ref = _sdpa_reference(_f64(q[s:s + 1]), _f64(seqs_k[s]), _f64(seqs_v[s]), G,
                              head_map=list(hmap))
        np.testing.assert_allclose(out[s:s + 1], ref, rtol=0, atol=1e-12)


def test_explicit_scale_matches_sdpa(oracle_mod):
    rng = np.random.default_rng(8)
    seqs_k = [_bf16(rng.standard_normal((21, 1, 8)))]
    seqs_v = [_bf16(rng.standard_normal((21, 1, 8)))]
    kp, vp, tables, cl = _pool_from_contiguous(oracle_mod, rng, seqs_k, seqs_v, 8)
    q = _bf16(rng.standard_normal((1, 2, 8)))
    qs = np.array([0, 1], np.int32)
    out = oracle_mod.paged_attention(kp, vp, q, qs, tables, cl, scale=0.3)
    ref = _sdpa_reference(_f64(q), _f64(seqs_k[0]), _f64(seqs_v[0]), 2, scale=0.3)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    default = oracle_mod.paged_attention(kp, vp, q, qs, tables, cl)
    explicit = oracle_mod.paged_attention(kp, vp, q, qs, tables, cl, scale=1 / math.sqrt(8))
    assert np.array_equal(default, explicit)


def _single_seq_pool(k_rows, v_rows, B=4, perm_seed=0):
    """Pool holding one sequence's rows [L, 1, D] in shuffled physical blocks."""
    L, H, D = k_rows.shape
    nb = (L + B - 1) // B
    perm = np.random.default_rng(perm_seed).permutation(nb + 2).astype(np.int32)
    kp = np.zeros((nb + 2, H, B, D), np.uint16)
    vp = np.zeros_like(kp)
    for t in range(L):
        kp[perm[t // B], :, t % B] = k_rows[t]
        vp[perm[t // B], :, t % B] = v_rows[t]
    return kp, vp, perm[:nb][None, :].copy(), np.array([L], np.int32)


def test_one_hot_key_reproduces_its_value_row(oracle_mod):
    rng = np.random.default_rng(3)
    L, D, j = 37, 16, 22
    K = np.zeros((L, 1, D), np.float32)
    K[:, 0, 0] = -1.0
    K[j, 0, 0] = 1.0
    V = _bf16(rng.standard_normal((L, 1, D)))
    kp, vp, tab, cl = _single_seq_pool(_bf16(K), V)
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 256.0                           # scores +-64 after 1/sqrt(16)
    out = oracle_mod.paged_attention(kp, vp, _bf16(q), np.array([0, 1], np.int32), tab, cl)
    np.testing.assert_allclose(out[0, 0], _f64(V[j, 0]), rtol=0, atol=1e-12)


def test_equal_keys_give_mean_value_and_single_token_gives_its_row(oracle_mod):
    rng = np.random.default_rng(4)
    L, D = 29, 8
    k0 = _bf16(rng.standard_normal((1, 1, D)))
    K = np.repeat(k0, L, axis=0)
    V = _bf16(rng.standard_normal((L, 1, D)))
    kp, vp, tab, cl = _single_seq_pool(K, V)
    q = _bf16(rng.standard_normal((1, 1, D)))
    out = oracle_mod.paged_attention(kp, vp, q, np.array([0, 1], np.int32), tab, cl)
    np.testing.assert_allclose(out[0, 0], _f64(V[:, 0]).mean(axis=0), rtol=0, atol=1e-12)
    out1 = oracle_mod.paged_attention(kp, vp, q, np.array([0, 1], np.int32), tab,
                                      np.array([1], np.int32))
    np.testing.assert_allclose(out1[0, 0], _f64(V[0, 0]), rtol=0, atol=0)


def test_sink_closed_form_and_vanishing_sink(oracle_mod):
    rng = np.random.default_rng(5)
    L, D = 11, 8
    K = _bf16(rng.standard_normal((L, 1, D)))
    V = _bf16(rng.standard_normal((L, 1, D)))
    kp, vp, tab, cl = _single_seq_pool(K, V)
    qs = np.array([0, 1], np.int32)
    q0 = np.zeros((1, 2, D), np.uint16)          # q = 0: every score is exactly 0
    sinks = np.array([0.7, -1.3], np.float32)
    out = oracle_mod.paged_attention(kp, vp, q0, qs, tab, cl, sinks=sinks)
    vsum = _f64(V[:, 0]).sum(axis=0)
    for h in range(2):
        expect = vsum / (L + math.exp(float(sinks[h])))
        np.testing.assert_allclose(out[0, h], expect, rtol=0, atol=1e-12)
    q = _bf16(rng.standard_normal((1, 2, D)))
    plain = oracle_mod.paged_attention(kp, vp, q, qs, tab, cl)
    tiny = oracle_mod.paged_attention(kp, vp, q, qs, tab, cl,
                                      sinks=np.full(2, -1e30, np.float32))
    assert np.array_equal(plain, tiny)
    big = oracle_mod.paged_attention(kp, vp, q, qs, tab, cl, sinks=np.full(2, 1e4, np.float32))
    assert np.all(np.abs(big) < 1e-300 + 1e-12)


def test_golden_uniform_scores_fixture(oracle_mod):
    fx = {}
    for line in open(os.path.join(GOLDEN, "attention_uniform_scores.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            key, _, rest = line.partition(" ")
            fx[key] = rest
    B = int(fx["block_size"])
    D = int(fx["head_dim"])
    table = np.array([[int(x) for x in fx["block_table"].split()]], np.int32)
    L = int(fx["context_len"])
    vrows = [[float(x) for x in r.split()] for r in fx["v_rows"].split("|")]
    nb = table.max() + 1
    kp = np.zeros((nb, 1, B, D), np.uint16)
    vp = np.zeros((nb, 1, B, D), np.uint16)
    for t in range(L):
        vp[table[0, t // B], 0, t % B] = _bf16(vrows[t])
        kp[table[0, t // B], 0, t % B] = _bf16(np.random.default_rng(t).standard_normal(D))
    q = np.zeros((1, 1, D), np.uint16)
    qs = np.array([0, 1], np.int32)
    cl = np.array([L], np.int32)
    out = oracle_mod.paged_attention(kp, vp, q, qs, table, cl)
    np.testing.assert_allclose(out[0, 0], [float(x) for x in fx["expect_no_sink"].split()], atol=1e-14)
    out = oracle_mod.paged_attention(kp, vp, q, qs, table, cl, sinks=np.zeros(1, np.float32))
    np.testing.assert_allclose(out[0, 0], [float(x) for x in fx["expect_sink_zero"].split()], atol=1e-14)


def test_physical_block_permutation_invariance(oracle_mod):
    b = wl.make_workload("tiny_decode", seed=11)
    k, v = b.k_pool[0].copy(), b.v_pool[0].copy()
    oracle_mod.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts,
                               b.k_new[0], b.v_new[0])
    out = oracle_mod.paged_attention(k, v, b.q[0], b.q_starts, b.block_tables, b.context_lens)
    perm = np.random.default_rng(0).permutation(b.num_blocks)   # new id of old block i = perm[i]
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    tables2 = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    out2 = oracle_mod.paged_attention(k2, v2, b.q[0], b.q_starts, tables2, b.context_lens)
    assert np.array_equal(out, out2)


def test_shared_prefix_blocks_equal_duplicated_blocks(oracle_mod):
    S, prefix = 5, 37
    lens = np.array([50, 41, 70, 38, 90])
    sharing = np.array([True, True, False, True, True])
    b = wl.build_batch(99, name="share", lens=lens, n_new=np.zeros(S, np.int64),
                       q_rows=np.ones(S, np.int64), num_q_heads=4, num_kv_heads=2, head_dim=16,
                       block_size=8, causal=False, shared_prefix=prefix, sharing=sharing)
    assert len(b.shared_block_ids) == prefix // 8
    k, v = b.k_pool[0], b.v_pool[0]
    out = oracle_mod.paged_attention(k, v, b.q[0], b.q_starts, b.block_tables, b.context_lens)
    # give every sharing sequence its own private copy of the shared blocks
    nsh = len(b.shared_block_ids)
    n_sharing = int(sharing.sum())
    extra = nsh * n_sharing
    k2 = np.concatenate([k, np.zeros((extra,) + k.shape[1:], np.uint16)])
    v2 = np.concatenate([v, np.zeros((extra,) + v.shape[1:], np.uint16)])
    tables2 = b.block_tables.copy()
    nxt = b.num_blocks
    for s in np.nonzero(sharing)[0]:
        for j in range(nsh):
            src = b.block_tables[s, j]
            k2[nxt] = k[src]
            v2[nxt] = v[src]
            tables2[s, j] = nxt
            nxt += 1
    out2 = oracle_mod.paged_attention(k2, v2, b.q[0], b.q_starts, tables2, b.context_lens)
    assert np.array_equal(out, out2)


def test_causal_window_row_equals_decode_over_its_prefix(oracle_mod):
    S = 3
    lens = np.array([40, 23, 65])
    W = np.array([6, 1, 16])
    b = wl.build_batch(5, name="win", lens=lens, n_new=W, q_rows=W, num_q_heads=4,
                       num_kv_heads=2, head_dim=16, block_size=8, causal=True)
    k, v = b.k_pool[0].copy(), b.v_pool[0].copy()
    oracle_mod.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts,
                               b.k_new[0], b.v_new[0])
    out = oracle_mod.paged_attention(k, v, b.q[0], b.q_starts, b.block_tables, b.context_lens,
                                     causal=True)
    for s in range(S):
        for w in range(W[s]):
            r = b.q_starts[s] + w
            one = oracle_mod.paged_attention(
                k, v, b.q[0][r:r + 1], np.array([0, 1], np.int32), b.block_tables[s:s + 1],
                np.array([lens[s] - W[s] + w + 1], np.int32), causal=False)
            assert np.array_equal(out[r], one[0])


def test_row_without_keys_outputs_zero(oracle_mod):
    kp = np.zeros((2, 1, 4, 8), np.uint16)
    vp = np.full((2, 1, 4, 8), 0x3F80, np.uint16)
    q = _bf16(np.ones((1, 2, 8)))
    tab = np.array([[0]], np.int32)
    out = oracle_mod.paged_attention(kp, vp, q, np.array([0, 1], np.int32), tab,
                                     np.array([0], np.int32))
    assert np.all(out == 0)
    out = oracle_mod.paged_attention(kp, vp, q, np.array([0, 1], np.int32), tab,
                                     np.array([0], np.int32), sinks=np.zeros(2, np.float32))
    assert np.all(out == 0)


def test_rejects_bad_block_ids_and_head_maps(oracle_mod):
    kp = np.zeros((2, 1, 4, 8), np.uint16)
    q = np.zeros((1, 2, 8), np.uint16)
    qs = np.array([0, 1], np.int32)
    with pytest.raises(ValueError):
        oracle_mod.paged_attention(kp, kp, q, qs, np.array([[5]], np.int32), np.array([3], np.int32))
    with pytest.raises(ValueError):
        oracle_mod.paged_attention(kp, kp, q, qs, np.array([[0]], np.int32), np.array([9], np.int32))
    with pytest.raises(ValueError):
        oracle_mod.paged_attention(kp, kp, q, qs, np.array([[0]], np.int32), np.array([3], np.int32),
                                   kv_head_of_q_head=np.array([0, 1], np.int32))
