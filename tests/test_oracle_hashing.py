"""Oracle pins for the chained content keys of full KV blocks.

TensorSharp "高级功能", section "连续批处理与分页 KV 缓存": every full block is
content-hashed so identical prefixes share blocks.  The primitives are pinned by
their published test vectors; the chaining by the invariants prefix sharing
needs (equal prefixes -> equal keys, a change anywhere -> every later key
changes, partial blocks never keyed, a continued chain equals the whole chain).
"""
import pathlib

import numpy as np
import pytest

GOLDEN = pathlib.Path(__file__).parent / "golden" / "hash_vectors.txt"


def _golden():
    fnv, sm = [], []
    for line in GOLDEN.read_text().splitlines():
        if line.startswith("fnv1a64 "):
            _, rest = line.split(" ", 1)
            text, digest = rest.rsplit(" ", 1)
            fnv.append((text.strip('"').encode(), int(digest, 16)))
        elif line.startswith("splitmix64 "):
            parts = line.split()[1:]
            sm.append((int(parts[0]), [int(x) for x in parts[1:]]))
    return fnv, sm


def test_fnv1a64_published_vectors(oracle_mod):
    fnv, _ = _golden()
    assert len(fnv) == 3
    for data, digest in fnv:
        assert oracle_mod.fnv1a64(data) == digest


def test_splitmix64_published_stream(oracle_mod):
    _, sm = _golden()
    (seed, outs), = sm
    state = seed
    got = []
    for _ in outs:
        state = (state + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        got.append(oracle_mod.splitmix64_mix(state))
    assert got == outs


def _seqs(rng, lens, vocab=50000):
    toks = [rng.integers(0, vocab, size=n, dtype=np.int32) for n in lens]
    starts = np.zeros(len(lens) + 1, dtype=np.int32)
    starts[1:] = np.cumsum(lens)
    return toks, starts


def test_block_key_is_mix_of_fnv_over_little_endian_ids(oracle_mod):
    # glue between the pinned primitives: byte order from numpy's '<i4' encoding
    rng = np.random.default_rng(1)
    toks = rng.integers(-2**31, 2**31 - 1, size=48, dtype=np.int64).astype(np.int32)
    starts = np.array([0, 48], dtype=np.int32)
    seed = 0x0123456789ABCDEF
    keys = oracle_mod.block_hashes(toks, starts, 16, seed, 4)
    h = seed
    for i in range(3):
        c = oracle_mod.fnv1a64(toks[16 * i:16 * i + 16].astype("<i4").tobytes())
        h = oracle_mod.splitmix64_mix(h ^ c)
        assert int(keys[0, i]) == h
    assert int(keys[0, 3]) == 0


def test_equal_prefixes_share_keys_and_divergence_propagates(oracle_mod):
    rng = np.random.default_rng(2)
    B = 16
    base = rng.integers(0, 50000, size=10 * B + 5, dtype=np.int32)
    a = base.copy()
    b = base.copy()
    b[4 * B + 3] += 1                        # differs in block 4 only
    c = base[: 7 * B + 9].copy()             # shorter: 7 full blocks, a partial one
    toks = np.concatenate([a, b, c])
    starts = np.array([0, len(a), len(a) + len(b), len(toks)], dtype=np.int32)
    keys = oracle_mod.block_hashes(toks, starts, B, 99, 12)
    assert np.array_equal(keys[0, :4], keys[1, :4])
    assert np.all(keys[0, 4:10] != keys[1, 4:10])           # every later key changes
    assert np.array_equal(keys[2, :7], keys[0, :7])
    assert np.all(keys[0, :10] != 0) and np.all(keys[0, 10:] == 0)   # partial block 10 unkeyed
    assert np.all(keys[2, 7:] == 0)
    # the same block contents at another position get another key (prefix differs)
    rep = np.tile(base[:B], 3)
    k2 = oracle_mod.block_hashes(rep, np.array([0, 3 * B], np.int32), B, 99, 3)
    assert len(set(int(x) for x in k2[0])) == 3


def test_seed_changes_every_key(oracle_mod):
    rng = np.random.default_rng(3)
    toks, starts = _seqs(rng, [64])
    k1 = oracle_mod.block_hashes(toks[0], starts, 16, 1, 4)
    k2 = oracle_mod.block_hashes(toks[0], starts, 16, 2, 4)
    assert np.all(k1 != k2)


def test_continued_chain_equals_whole_chain(oracle_mod):
    rng = np.random.default_rng(4)
    B = 16
    lens = [5 * B + 3, 9 * B, 2 * B + 15]
    toks, starts = _seqs(rng, lens)
    whole = oracle_mod.block_hashes(np.concatenate(toks), starts, B, 7, 10)
    # hash the first 2 blocks, then continue from the second key with the rest
    first = [t[: 2 * B] for t in toks]
    rest = [t[2 * B:] for t in toks]
    fs = np.array([0] + list(np.cumsum([len(x) for x in first])), np.int32)
    rs = np.array([0] + list(np.cumsum([len(x) for x in rest])), np.int32)
    k1 = oracle_mod.block_hashes(np.concatenate(first), fs, B, 7, 10)
    k2 = oracle_mod.block_hashes(np.concatenate(rest), rs, B, 0, 10, chain_in=k1[:, 1].copy())
    for s, n in enumerate(lens):
        full = n // B
        assert np.array_equal(whole[s, :2], k1[s, :2])
        assert np.array_equal(whole[s, 2:full], k2[s, : full - 2])


def test_empty_and_short_sequences(oracle_mod):
    toks = np.arange(20, dtype=np.int32)
    starts = np.array([0, 0, 15, 20], dtype=np.int32)
    keys = oracle_mod.block_hashes(toks, starts, 16, 5, 2)
    assert np.all(keys == 0)
    with pytest.raises(ValueError):
        oracle_mod.block_hashes(np.arange(40, dtype=np.int32), np.array([0, 40], np.int32), 16, 5, 1)
