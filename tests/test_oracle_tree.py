"""Pins for the oracle's tree verify (attention with per-row ancestor masks) and tree accept.

TensorFold article, section "接受规则：GPU 上的 accept 内核": verify rows form a chain or a tree;
each row attends to the cached context and its own ancestors; the accepted path follows the
child whose token equals the target's choice.
"""
import itertools
import os

import numpy as np
import pytest
import torch

from paged_kv_attention_forward_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    fx = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            key, _, rest = line.partition(" ")
            fx[key] = [int(x) for x in rest.split()]
    return fx


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def random_tree_parents(rng, W):
    return np.array([-1] + [int(rng.integers(0, j)) for j in range(1, W)], np.int32)


def ancestor_masks(parents):
    W = len(parents)
    masks = np.zeros(W, np.uint32)
    for j in range(W):
        m, u = 0, j
        while u >= 0:
            m |= 1 << u
            u = parents[u] if u > 0 else -1
        masks[j] = m
    return masks


def test_chain_masks_equal_causal_window(oracle_mod):
    lens = np.array([40, 23, 65])
    W = np.array([6, 1, 16])
    b = wl.build_batch(3, name="chain", lens=lens, n_new=np.zeros(3, np.int64), q_rows=W, num_q_heads=4,
                       num_kv_heads=2, head_dim=16, block_size=8, causal=True)
    masks = np.concatenate([(1 << (np.arange(w) + 1)) - 1 for w in W]).astype(np.uint32)
    args = (b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables, b.context_lens)
    causal = oracle_mod.paged_attention(*args, causal=True)
    tree = oracle_mod.paged_attention(*args, tree_masks=masks)
    assert np.array_equal(causal, tree)


@pytest.mark.parametrize("shape", ["tree", "arbitrary"])
def test_tree_masks_match_sdpa_with_explicit_mask(oracle_mod, shape):
    rng = np.random.default_rng(11)
    lens = np.array([30, 57])
    W = np.array([7, 12])
    b = wl.build_batch(4, name="tree", lens=lens, n_new=np.zeros(2, np.int64), q_rows=W, num_q_heads=6,
                       num_kv_heads=2, head_dim=16, block_size=8, causal=False)
    if shape == "tree":
        parents = [random_tree_parents(rng, w) for w in W]
        masks = np.concatenate([ancestor_masks(p) for p in parents]).astype(np.uint32)
    else:   # any bit pattern, including ones that hide window token 0
        masks = rng.integers(0, 1 << 12, size=int(W.sum())).astype(np.uint32)
    out = oracle_mod.paged_attention(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables,
                                     b.context_lens, tree_masks=masks)
    G, B = 3, 8
    for s in range(2):
        L, w_s = int(lens[s]), int(W[s])
        t = np.arange(L)
        K = np.stack([b.k_pool[0][b.block_tables[s, i // B], :, i % B] for i in t])
        V = np.stack([b.v_pool[0][b.block_tables[s, i // B], :, i % B] for i in t])
        rows = slice(b.q_starts[s], b.q_starts[s + 1])
        vis = np.zeros((w_s, L), bool)
        for w in range(w_s):
            m = int(masks[b.q_starts[s] + w])
            vis[w] = (t < L - w_s) | ((t >= L - w_s) & (((m >> np.maximum(t - (L - w_s), 0)) & 1) == 1))
        Q = torch.from_numpy(_f64(b.q[0][rows])).permute(1, 0, 2)
        Kx = torch.from_numpy(_f64(K)[:, [h // G for h in range(6)], :]).permute(1, 0, 2)
        Vx = torch.from_numpy(_f64(V)[:, [h // G for h in range(6)], :]).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(Q[None], Kx[None], Vx[None],
                                                               attn_mask=torch.from_numpy(vis))
        np.testing.assert_allclose(out[rows], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_golden_tree_accept(oracle_mod):
    fx = _fixture("accept_tree_worked_example.txt")
    V = fx["vocab"][0]
    for suf in ("", "2"):
        am = np.array(fx["argmax" + suf], np.int32)
        lg = np.zeros((len(am), V), np.float32)
        lg[np.arange(len(am)), am] = 1.0
        got = oracle_mod.spec_accept_tree_greedy(lg, np.array([0, len(am)], np.int32),
                                                 np.array(fx["drafts" + suf], np.int32),
                                                 np.array(fx["parents" + suf], np.int32))
        assert np.array_equal(got[0], am)
        assert got[1][0] == fx["expect_accept_len" + suf][0]
        assert got[2].tolist() == fx["expect_out_tokens" + suf]
        assert got[3].tolist() == fx["expect_accepted_rows" + suf]


def test_tree_accept_on_chains_equals_chain_accept(oracle_mod):
    b = wl.make_workload("spec_verify", seed=3)
    parents = np.concatenate([np.arange(-1, w - 1) for w in np.diff(b.q_starts)]).astype(np.int32)
    a1, n1, o1 = oracle_mod.spec_accept_greedy(b.logits, b.q_starts, b.draft_tokens)
    a2, n2, o2, rows = oracle_mod.spec_accept_tree_greedy(b.logits, b.q_starts, b.draft_tokens, parents)
    assert np.array_equal(a1, a2) and np.array_equal(n1, n2) and np.array_equal(o1, o2)
    for s in range(b.num_seqs):
        r0 = b.q_starts[s]
        assert rows[r0:r0 + n2[s]].tolist() == list(range(1, n2[s] + 1))


def test_tree_accept_brute_force_small_trees(oracle_mod):
    """Every tree shape with 1..4 nodes, drafts and targets over a 2-token vocabulary.
    Checked property: the accepted nodes form a root path whose every step picks the
    lowest-index child carrying the parent's target token, and the last node has no
    child carrying its target token."""
    V = 2
    for W in range(1, 5):
        shapes = itertools.product(*[range(j) for j in range(1, W)])
        for par in shapes:
            parents = np.array([-1, *par], np.int32)
            for am in itertools.product(range(V), repeat=W):
                for dr in itertools.product(range(V), repeat=W - 1):
                    drafts = np.array([-1, *dr], np.int32)
                    lg = np.zeros((W, V), np.float32)
                    lg[np.arange(W), am] = 1.0
                    a, n, out, rows = oracle_mod.spec_accept_tree_greedy(lg, np.array([0, W], np.int32),
                                                                         drafts, parents)
                    n = int(n[0])
                    path = [0] + rows[:n].tolist()
                    for u, c in zip(path, path[1:]):
                        kids = [k for k in range(1, W) if parents[k] == u and drafts[k] == am[u]]
                        assert kids and c == kids[0]
                    last = path[-1]
                    assert not [k for k in range(1, W) if parents[k] == last and drafts[k] == am[last]]
                    assert out[:n].tolist() == [int(drafts[c]) for c in path[1:]]
                    assert out[n] == am[last] and np.all(out[n + 1:] == -1) and np.all(rows[n:] == -1)


def test_tree_accept_rejects_bad_parents(oracle_mod):
    lg = np.eye(3, dtype=np.float32)
    with pytest.raises(ValueError):
        oracle_mod.spec_accept_tree_greedy(lg, np.array([0, 3], np.int32), np.array([-1, 0, 1], np.int32),
                                           np.array([-1, 0, 2], np.int32))
