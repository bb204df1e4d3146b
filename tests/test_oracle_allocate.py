"""Pins for the oracle's block allocator with prefix sharing (no GPU).

TensorSharp "高级功能", section "连续批处理与分页 KV 缓存": KV blocks of a fixed size come
from one shared pool; every full block is content-hashed so that identical prefixes map to
the same physical blocks; a partial block is never shared.  The oracle states the
allocation as the sequential engine step (sequences in order, blocks in order, the free
stack popped from its top).  Pinned here by a worked example done by hand, by brute-force
properties on random batches (which entries share a block, reference counts, pop order),
by invariance of the sharing structure to the order of the sequences, and by the attention
over tables it builds equalling the attention over the workload's own tables.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EMPTY = np.uint64(0xFFFFFFFFFFFFFFFF)


def _read_golden():
    g = {"keys": {}, "table": {}, "fresh": {}, "table_before": {}}
    for line in open(os.path.join(GOLDEN, "block_allocate_worked_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = line.split()
        if w[0] in ("keys",):
            g["keys"][int(w[1])] = [int(x, 16) for x in w[2:]]
        elif w[0] in ("table", "fresh"):
            g[w[0]][int(w[1])] = [-1 if x == "-" else int(x) for x in w[2:]]
        elif w[0] == "table_before":
            g["table_before"][(int(w[1]), int(w[2]))] = int(w[3])
        elif w[0] in ("index_before", "index_after"):
            g[w[0]] = {int(k, 16): (int(i), int(r)) for k, i, r in (x.split(":") for x in w[1:])}
        else:
            g[w[0]] = [int(x) for x in w[1:]]
    return g


def test_worked_example(oracle_mod):
    g = _read_golden()
    S, mb = len(g["lens"]), g["max_blocks"][0]
    keys = np.array([g["keys"][s] for s in range(S)], np.uint64)
    tables = np.full((S, mb), -1, np.int32)
    for (s, j), v in g["table_before"].items():
        tables[s, j] = v
    ib = g["index_before"]
    ix = oracle_mod.BlockIndex(list(ib), [v[0] for v in ib.values()], [v[1] for v in ib.values()])
    fids = np.array(g["free_ids"], np.int32)
    new_ix, t, fresh, fc, bits = oracle_mod.block_allocate(ix, fids, len(fids), keys, g["lens"],
                                                           g["first_block"], g["block_size"][0], tables)
    assert t.tolist() == [g["table"][s] for s in range(S)]
    assert fresh.tolist() == [g["fresh"][s] for s in range(S)]
    assert new_ix.as_dict() == g["index_after"]
    assert fc == g["free_count_after"][0] and bits == g["status"][0]


def test_exhaustion_and_a_failed_key(oracle_mod):
    # two new keys and a private block but one free block: the first pop succeeds, the rest
    # give -1 and set bit 128; the failed key's later occurrence gets -1 without a pop
    keys = np.array([[5, 6, 0], [6, 0, 0]], np.uint64)
    ix, t, fresh, fc, bits = oracle_mod.block_allocate(oracle_mod.BlockIndex(), [40], 1, keys, [9, 4], [0, 0], 4,
                                                       np.full((2, 3), -1, np.int32))
    assert t.tolist() == [[40, -1, -1], [-1, -1, -1]]
    assert fresh.tolist() == [[1, 0, 0], [0, 0, 0]]
    assert ix.as_dict() == {5: (40, 1), 6: (-1, 0)} and fc == 0 and bits == 128
    # a later call with blocks to spare allocates the failed key (its entry had no block)
    ix2, t2, fresh2, fc2, bits2 = oracle_mod.block_allocate(ix, [50, 51], 2, np.array([[6]], np.uint64), [4], [0],
                                                            4, np.full((1, 1), -1, np.int32))
    assert t2.tolist() == [[51]] and fresh2.tolist() == [[1]] and ix2.as_dict()[6] == (51, 1) and bits2 == 0


def test_empty_key_and_overrun(oracle_mod):
    # a full block whose key is the reserved empty key is private; a length past the table
    # is cut to max_blocks and flagged (bit 2)
    keys = np.array([[EMPTY, EMPTY]], np.uint64)
    ix, t, fresh, fc, bits = oracle_mod.block_allocate(oracle_mod.BlockIndex(), [1, 2, 3], 3, keys, [13], [0], 4,
                                                       np.full((1, 2), -1, np.int32))
    assert t.tolist() == [[3, 2]] and fresh.tolist() == [[1, 1]] and len(ix.keys) == 0
    assert bits == 2 and fc == 1


def _random_case(rng, S=12, mb=9, B=4, n_keys=15, F=200):
    keys = rng.integers(0, n_keys, size=(S, mb)).astype(np.uint64) + np.uint64(100)
    lens = rng.integers(0, mb * B + 1, size=S).astype(np.int32)
    first = np.array([rng.integers(0, max(1, -(-int(L) // B)) + 1) for L in lens], np.int32)
    tables = np.full((S, mb), -3, np.int32)
    free_ids = rng.permutation(1000)[:F].astype(np.int32)
    pre = oracle_index = None
    pre_keys = rng.choice(n_keys, size=4, replace=False).astype(np.uint64) + np.uint64(100)
    pre = (pre_keys, np.array([900, 901, 902, 903], np.int32), np.array([1, 2, 1, 5], np.int32))
    return keys, lens, first, tables, free_ids, pre, B


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_properties(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    keys, lens, first, tables, free_ids, pre, B = _random_case(rng)
    S, mb = keys.shape
    ix0 = oracle_mod.BlockIndex(*pre)
    ix, t, fresh, fc, bits = oracle_mod.block_allocate(ix0, free_ids, len(free_ids), keys, lens, first, B, tables)
    assert bits == 0
    alloc = []                                   # (s, j, keyed?, key) of every entry this call allocated
    for s in range(S):
        nb, nk = -(-int(lens[s]) // B), int(lens[s]) // B
        for j in range(mb):
            if j < first[s] or j >= nb:
                assert t[s, j] == -3 and fresh[s, j] == 0          # untouched
            else:
                alloc.append((s, j, j < nk, int(keys[s, j]) if j < nk else None))
    # two allocated entries name the same block iff both are full blocks with equal keys
    for a in range(len(alloc)):
        for b in range(a + 1, len(alloc)):
            sa, ja, ka, xa = alloc[a]
            sb, jb, kb, xb = alloc[b]
            assert (t[sa, ja] == t[sb, jb]) == (ka and kb and xa == xb), (alloc[a], alloc[b])
    # pops: one per new key plus one per private block, taken from the stack's top in order
    pre_keys = set(int(k) for k in pre[0])
    new_keys, order = [], []
    for s, j, keyed, key in alloc:
        if not keyed:
            order.append((s, j))
        elif key not in pre_keys and key not in new_keys:
            new_keys.append(key)
            order.append((s, j))
    popped = [int(t[s, j]) for s, j in order]
    assert popped == [int(x) for x in free_ids[::-1][:len(order)]]
    assert fc == len(free_ids) - len(order)
    assert [int(fresh[s, j]) for s, j, *_ in alloc] == [int((s, j) in order) for s, j, *_ in alloc]
    # reference counts: earlier count + one per table entry of this call naming the key
    d = ix.as_dict()
    for k, (i, r) in d.items():
        before = dict(zip(map(int, pre[0]), map(int, pre[2]))).get(k, 0)
        uses = sum(1 for s, j, keyed, key in alloc if keyed and key == k)
        assert r == before + uses
        if k in pre_keys:
            assert i == dict(zip(map(int, pre[0]), map(int, pre[1])))[k]


@pytest.mark.parametrize("seed", range(4))
def test_sharing_structure_does_not_depend_on_sequence_order(oracle_mod, seed):
    """Which table entries share a block, the reference counts and the number of pops are
    the same whatever order the sequences come in; only which free block goes where moves."""
    rng = np.random.default_rng(50 + seed)
    keys, lens, first, tables, free_ids, pre, B = _random_case(rng)
    perm = rng.permutation(len(lens))
    a = oracle_mod.block_allocate(oracle_mod.BlockIndex(*pre), free_ids, len(free_ids), keys, lens, first, B, tables)
    b = oracle_mod.block_allocate(oracle_mod.BlockIndex(*pre), free_ids, len(free_ids), keys[perm], lens[perm],
                                  first[perm], B, tables[perm])
    ta, tb = a[1], b[1][np.argsort(perm)]
    fa, fb = a[2], b[2][np.argsort(perm)]
    assert a[3] == b[3]                                               # pops
    assert {k: v[1] for k, v in a[0].as_dict().items()} == {k: v[1] for k, v in b[0].as_dict().items()}
    pos = [(s, j) for s in range(ta.shape[0]) for j in range(ta.shape[1]) if ta[s, j] != -3]
    assert pos == [(s, j) for s in range(tb.shape[0]) for j in range(tb.shape[1]) if tb[s, j] != -3]
    for x in range(len(pos)):
        for y in range(x + 1, len(pos)):
            assert (ta[pos[x]] == ta[pos[y]]) == (tb[pos[x]] == tb[pos[y]])
    assert int(fa.sum()) == int(fb.sum())


def test_tables_it_builds_give_the_same_attention(oracle_mod):
    """A shared-prefix batch: token ids -> chained block keys -> allocation from an empty
    index; every fresh block is filled with the K/V its tokens hold in the workload's own
    pool.  Attention through the new tables equals attention through the workload's tables
    exactly (the float64 oracle walks the same values in the same order)."""
    from paged_kv_attention_forward_gb300 import workloads as wl
    b = wl.make_workload("cb_mix", seed=3, num_seqs=8)
    B, mb = b.block_size, b.max_blocks_per_seq
    toks, starts = wl.context_token_ids(b, seed=4)
    keys = oracle_mod.block_hashes(toks, starts, B, 77, mb)
    keys[keys == 0] = EMPTY                      # rows past the full blocks carry no key
    nb_pool = b.num_blocks
    free_ids = np.random.default_rng(5).permutation(nb_pool).astype(np.int32)
    S = b.num_seqs
    ix, t, fresh, fc, bits = oracle_mod.block_allocate(oracle_mod.BlockIndex(), free_ids, nb_pool, keys,
                                                       b.context_lens, np.zeros(S, np.int32), B,
                                                       np.full((S, mb), -1, np.int32))
    assert bits == 0
    # the shared prefix's full blocks map to one block each, shared by every sharing sequence
    full_shared = b.shared_prefix // B
    s0 = b.sharing_seqs[0]
    for s in b.sharing_seqs[1:]:
        assert np.array_equal(t[s, :full_shared], t[s0, :full_shared])
    assert fresh.sum() < sum(-(-int(L) // B) for L in b.context_lens)
    k_new = np.full_like(b.k_pool[0], 0x7FC0)    # bf16 NaN in every block nobody fills
    v_new = np.full_like(b.v_pool[0], 0x7FC0)
    for s in range(S):
        for j in range(-(-int(b.context_lens[s]) // B)):
            if fresh[s, j]:
                k_new[t[s, j]] = b.k_pool[0][b.block_tables[s, j]]
                v_new[t[s, j]] = b.v_pool[0][b.block_tables[s, j]]
    ref = oracle_mod.paged_attention(b.k_pool[0], b.v_pool[0], b.q[0], b.q_starts, b.block_tables, b.context_lens)
    got = oracle_mod.paged_attention(k_new, v_new, b.q[0], b.q_starts, t, b.context_lens)
    assert np.array_equal(got, ref)
