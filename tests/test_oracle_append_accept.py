"""Pins for the oracle's paged K/V append and greedy accept (no GPU).

Append follows TensorSharp "高级功能", section "连续批处理与分页 KV 缓存" and the
"批量前向" paragraph (new K/V scattered into paged slots; only full blocks are
hashed and shared).  Accept follows the TensorFold article, section
"接受规则：GPU 上的 accept 内核", and TensorSharp's "MTP / NextN 推测解码" section.
"""
import itertools
import os

import numpy as np

from paged_kv_attention_forward_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    fx = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            key, _, rest = line.partition(" ")
            fx.setdefault(key, []).append(rest)
    return fx


def _bf16(x):
    return wl.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_golden_append_worked_example(oracle_mod):
    fx = _fixture("append_worked_example.txt")
    nb, B = int(fx["num_blocks"][0]), int(fx["block_size"][0])
    H, D = int(fx["num_kv_heads"][0]), int(fx["head_dim"][0])
    table = np.array([[int(x) for x in fx["block_table"][0].split()]], np.int32)
    old = np.array([int(fx["context_len_old"][0])], np.int32)
    krows = [[float(x) for x in r.split()] for r in fx["k_new"][0].split("|")]
    vrows = [[float(x) for x in r.split()] for r in fx["v_new"][0].split("|")]
    kn = _bf16(np.array(krows)[:, None, :])
    vn = _bf16(np.array(vrows)[:, None, :])
    kp = np.full((nb, H, B, D), 0x1234, np.uint16)
    vp = np.full((nb, H, B, D), 0x4321, np.uint16)
    k0, v0 = kp.copy(), vp.copy()
    oracle_mod.paged_kv_append(kp, vp, table, old, np.array([0, len(krows)], np.int32), kn, vn)
    touched = np.zeros((nb, B), bool)
    for e in fx["expect"]:
        tok = e.split()
        blk, slot = int(tok[1]), int(tok[3])
        kx = [float(tok[5]), float(tok[6])]
        vx = [float(tok[8]), float(tok[9])]
        assert np.array_equal(kp[blk, 0, slot], _bf16(kx))
        assert np.array_equal(vp[blk, 0, slot], _bf16(vx))
        touched[blk, slot] = True
    untouched = ~touched
    assert np.array_equal(kp[:, 0][untouched], k0[:, 0][untouched])
    assert np.array_equal(vp[:, 0][untouched], v0[:, 0][untouched])


def test_append_touches_exactly_the_new_slots_and_never_shared_blocks(oracle_mod):
    b = wl.make_workload("cb_mix", seed=3)
    k, v = b.k_pool[0].copy(), b.v_pool[0].copy()
    oracle_mod.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts,
                               b.k_new[0], b.v_new[0])
    changed = np.any(k != b.k_pool[0], axis=(1, 3)) | np.any(v != b.v_pool[0], axis=(1, 3))  # [nb, B]
    # a changed slot may coincide with equal filler bits; count slots that must change
    assert changed.sum() <= b.num_seqs
    assert not changed[b.shared_block_ids].any()
    # every appended row reads back at the position the cache length implies
    for s in range(b.num_seqs):
        p = int(b.context_lens_old[s])
        blk = b.block_tables[s, p // b.block_size]
        row = b.new_starts[s]
        assert np.array_equal(k[blk, :, p % b.block_size], b.k_new[0][row])
        assert np.array_equal(v[blk, :, p % b.block_size], b.v_new[0][row])


def test_argmax_matches_numpy_including_ties(oracle_mod):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((20, 1000)).astype(np.float32)
    x[3, [10, 500, 999]] = 50.0                      # three-way tie
    x[4, :] = 1.0                                    # all equal
    x[5, [0, 1]] = 9.0
    x[6, -1] = 99.0
    x[7, 7] = np.float32(-0.0)
    x[7, :] = -1.0
    x[7, [2, 9]] = 0.0
    x[7, 5] = np.float32(-0.0)                       # -0 == +0: lowest index wins
    got = oracle_mod.argmax_rows(x)
    assert np.array_equal(got, np.argmax(x, axis=1))
    assert got[3] == 10 and got[4] == 0 and got[5] == 0 and got[6] == 999 and got[7] == 2


def test_golden_accept_worked_example(oracle_mod):
    fx = _fixture("accept_worked_example.txt")
    V = int(fx["vocab"][0])

    def logits_for(am):
        lg = np.zeros((len(am), V), np.float32)
        lg[np.arange(len(am)), am] = 1.0
        return lg

    for suf in ("", "2", "3"):
        am = np.array([int(x) for x in fx["argmax" + suf][0].split()], np.int32)
        dr = np.array([int(x) for x in fx["drafts" + suf][0].split()], np.int32)
        a, n, out = oracle_mod.spec_accept_greedy(logits_for(am), np.array([0, len(am)], np.int32), dr)
        assert np.array_equal(a, am)
        assert n[0] == int(fx["expect_accept_len" + suf][0])
        assert np.array_equal(out, [int(x) for x in fx["expect_out_tokens" + suf][0].split()])
    row = np.array([[float(x) for x in fx["tie_row"][0].split()]], np.float32)
    assert oracle_mod.argmax_rows(row)[0] == int(fx["tie_argmax"][0])


def test_accept_brute_force_small_chains(oracle_mod):
    """All argmax paths and drafts over a 3-token vocabulary, windows of 1..4 rows.

    Checked property (the definition of the longest matching prefix): the emitted
    tokens are the target's own greedy tokens a_0..a_n, every accepted draft equals
    the previous row's target token, and the walk stops at the window end or at the
    first mismatching draft."""
    V = 3
    for W in range(1, 5):
        for am in itertools.product(range(V), repeat=W):
            for dr in itertools.product(range(V), repeat=W - 1):
                lg = np.zeros((W, V), np.float32)
                lg[np.arange(W), am] = 2.0
                for i in range(1, W, 2):                    # ties on odd rows
                    lg[i, (am[i] + 1) % V] = 2.0
                expect_am = np.argmax(lg, axis=1)
                drafts = np.array([-1] + list(dr), np.int32)
                a, n, out = oracle_mod.spec_accept_greedy(lg, np.array([0, W], np.int32), drafts)
                n = int(n[0])
                assert np.array_equal(a, expect_am)
                assert 0 <= n <= W - 1
                assert all(drafts[i] == a[i - 1] for i in range(1, n + 1))
                assert n == W - 1 or drafts[n + 1] != a[n]
                assert np.array_equal(out[:n + 1], a[:n + 1])
                assert np.all(out[n + 1:] == -1)


def test_accept_multiple_sequences_and_empty_sequence(oracle_mod):
    b = wl.make_workload("spec_verify", seed=2)
    a, n, out = oracle_mod.spec_accept_greedy(b.logits, b.q_starts, b.draft_tokens)
    assert np.array_equal(a, np.argmax(b.logits, axis=1))
    assert np.array_equal(a, b.planted_targets)      # the planted value is each row's maximum
    for s in range(b.num_seqs):
        r0, r1 = b.q_starts[s], b.q_starts[s + 1]
        one = oracle_mod.spec_accept_greedy(b.logits[r0:r1], np.array([0, r1 - r0], np.int32),
                                            b.draft_tokens[r0:r1])
        assert one[1][0] == n[s] and np.array_equal(one[2], out[r0:r1])
    qs = np.array([0, 2, 2, 3], np.int32)
    lg = np.eye(4, dtype=np.float32)[:3]
    a, n, out = oracle_mod.spec_accept_greedy(lg, qs, np.array([-1, 0, -1], np.int32))
    assert n.tolist() == [1, -1, 0] and out.tolist() == [0, 1, 2]
