"""GPU block allocation with prefix sharing against the oracle, bit-exact.

TensorSharp "高级功能", section "连续批处理与分页 KV 缓存": fixed-size blocks from one
shared pool; every full block is content-hashed so identical prefixes share physical
blocks; a partial block stays private.  The oracle states the sequential engine step; the
device call must give the same block tables, fresh flags, free-stack count and index
contents (key -> block id, reference count) whatever order its threads run in.  On a
shared-prefix batch at the continuous-batching config's size, the tables it builds must
give attention bit-identical to the workload's own tables.
"""
import numpy as np
import pytest

import oracle
from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import dev, dev_bf16, gpu_batch, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
EMPTY = np.uint64(0xFFFFFFFFFFFFFFFF)


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


def _keys_dev(keys):
    return dev(np.ascontiguousarray(keys, np.uint64).view(np.int64))


def _gpu_alloc(pkv, index, keys, lens, first, B, tables):
    t = dev(np.asarray(tables, np.int32))
    fresh = pkv.paged_block_allocate(index, _keys_dev(keys), dev(np.asarray(lens, np.int32)),
                                     dev(np.asarray(first, np.int32)), B, t)
    torch.cuda.synchronize()
    return t.cpu().numpy(), fresh.cpu().numpy(), int(index.free_count.item())


def _compare(pkv, index, ox, keys, lens, first, B, tables, free_ids, F, expect_bits=0):
    """One call on both sides: returns the oracle's index state for the next call."""
    t, fresh, fc = _gpu_alloc(pkv, index, keys, lens, first, B, tables)
    ox2, ot, ofresh, ofc, obits = oracle.block_allocate(ox, free_ids, F, keys, lens, first, B, tables)
    assert np.array_equal(t, ot), "block tables"
    assert np.array_equal(fresh, ofresh), "fresh flags"
    assert fc == ofc, "free count"
    assert index.entries() == ox2.as_dict(), "index contents"
    rc, bits = pkv.device_status()
    assert bits == expect_bits == obits, (rc, bits, obits)
    return ox2, ofc


def test_worked_example(pkv):
    # the hand-worked example of the oracle's pins, index state carried by a first call
    free_ids = np.arange(10, 18, dtype=np.int32)
    pre_free = np.array([3], np.int32)            # a first call puts key 0xA at block 3, refcount 2
    ix = pkv.BlockIndex(64, dev(np.concatenate([free_ids, pre_free])))
    ox = oracle.BlockIndex()
    keys0 = np.array([[0xA, 0], [0xA, 0]], np.uint64)
    allf = np.concatenate([free_ids, pre_free])
    ox, fc = _compare(pkv, ix, ox, keys0, [4, 4], [0, 0], 4, np.full((2, 2), -1, np.int32), allf, len(allf))
    assert ox.as_dict() == {0xA: (3, 2)} and fc == 8
    keys = np.zeros((4, 4), np.uint64)
    keys[0, :2] = [0xA, 0xB]
    keys[1, :2] = [0xA, 0xB]
    keys[2, :1] = [0x99]
    keys[3, :3] = [0xC, 0xB, 0xD]
    tables = np.full((4, 4), -1, np.int32)
    tables[2, 0] = 7
    ox, fc = _compare(pkv, ix, ox, keys, [10, 8, 5, 12], [0, 0, 1, 0], 4, tables, allf, fc)
    assert ox.as_dict() == {0xA: (3, 4), 0xB: (17, 3), 0xC: (14, 1), 0xD: (13, 1)} and fc == 3


@pytest.mark.parametrize("seed", range(4))
def test_random_calls_in_a_row(pkv, seed):
    """Three calls on one index: keys repeat within and across calls, some sequences keep
    allocated blocks (first_block > 0), lengths are ragged; a small index capacity makes
    probe chains long."""
    rng = np.random.default_rng(seed)
    free_ids = rng.permutation(5000).astype(np.int32)
    ix = pkv.BlockIndex(256, dev(free_ids))
    ox, fc = oracle.BlockIndex(), len(free_ids)
    B = [4, 16, 1][seed % 3]
    for call in range(3):
        S, mb = int(rng.integers(1, 40)), int(rng.integers(1, 12))
        keys = (rng.integers(0, 60, size=(S, mb)).astype(np.uint64) * np.uint64(0x9E3779B97F4A7C15))
        keys[rng.random((S, mb)) < 0.05] = EMPTY              # unindexable keys: private blocks
        lens = rng.integers(0, mb * B + 1, size=S).astype(np.int32)
        first = np.array([rng.integers(0, max(1, -(-int(L) // B)) + 1) for L in lens], np.int32)
        tables = rng.integers(-5, 0, size=(S, mb)).astype(np.int32)
        ox, fc = _compare(pkv, ix, ox, keys, lens, first, B, tables, free_ids, fc)


def test_running_out_of_blocks(pkv):
    rng = np.random.default_rng(7)
    free_ids = np.arange(100, 106, dtype=np.int32)           # six blocks for many more requests
    ix = pkv.BlockIndex(128, dev(free_ids))
    keys = rng.integers(0, 5, size=(6, 4)).astype(np.uint64) + np.uint64(11)
    lens = np.array([16, 13, 9, 16, 3, 11], np.int32)
    ox, fc = _compare(pkv, ix, oracle.BlockIndex(), keys, lens, np.zeros(6, np.int32), 4,
                      np.full((6, 4), -1, np.int32), free_ids, 6, expect_bits=128)
    assert fc == 0
    # more blocks arrive: the keys that got none are allocated on the next call
    more = np.arange(200, 240, dtype=np.int32)
    ix.free_ids = dev(more)
    ix.free_count.fill_(len(more))
    _compare(pkv, ix, ox, keys, lens, np.zeros(6, np.int32), 4, np.full((6, 4), -1, np.int32), more, len(more))


def _fill_from(b, t, fresh, k_pool, v_pool):
    """Copy every fresh block's contents from the workload's pool (through its own table)
    into the new pool at the allocated block (on the GPU)."""
    S = b.num_seqs
    src, dst = [], []
    for s in range(S):
        for j in range(-(-int(b.context_lens[s]) // b.block_size)):
            if fresh[s, j]:
                src.append(int(b.block_tables[s, j]))
                dst.append(int(t[s, j]))
    src_t = torch.tensor(src, dtype=torch.long, device="cuda")
    dst_t = torch.tensor(dst, dtype=torch.long, device="cuda")
    kn = torch.full_like(k_pool, float("nan"))
    vn = torch.full_like(v_pool, float("nan"))
    kn[dst_t] = k_pool[src_t]
    vn[dst_t] = v_pool[src_t]
    return kn, vn


def test_cb_mix_batch_built_through_the_allocator(pkv):
    """64 sequences, 48 sharing a 2900-token prefix: token ids -> paged_block_hashes ->
    paged_block_allocate from an empty index.  Tables, fresh flags and index bit-exact
    against the oracle; the 181 full prefix blocks are one physical block each; attention
    over a pool filled through the new tables equals attention over the workload's own
    tables bit for bit, including after a decode step's append allocates the next blocks."""
    b = wl.make_workload("cb_mix", seed=0)
    B, mb, S = b.block_size, b.max_blocks_per_seq, b.num_seqs
    g = gpu_batch(b)
    # the cached context first (lengths before the append), then the decode step's blocks
    toks, starts = wl.context_token_ids(b, seed=1)
    lens_old = b.context_lens_old
    starts_old = np.zeros(S + 1, np.int32)
    starts_old[1:] = np.cumsum(lens_old)
    toks_old = np.concatenate([toks[starts[s]:starts[s] + lens_old[s]] for s in range(S)])
    keys = pkv.paged_block_hashes(dev(toks_old), dev(starts_old), B, 99, mb)
    free_ids = np.random.default_rng(2).permutation(b.num_blocks).astype(np.int32)
    ix = pkv.BlockIndex(1 << 17, dev(free_ids))
    tables = torch.full((S, mb), -1, dtype=torch.int32, device="cuda")
    fresh = pkv.paged_block_allocate(ix, keys, dev(lens_old), dev(np.zeros(S, np.int32)), B, tables)
    torch.cuda.synchronize()
    keys_h = keys.cpu().numpy().view(np.uint64)
    ox, ot, ofresh, ofc, obits = oracle.block_allocate(oracle.BlockIndex(), free_ids, len(free_ids), keys_h,
                                                       lens_old, np.zeros(S, np.int32), B,
                                                       np.full((S, mb), -1, np.int32))
    t1, f1 = tables.cpu().numpy(), fresh.cpu().numpy()
    assert np.array_equal(t1, ot) and np.array_equal(f1, ofresh) and obits == 0
    assert ix.entries() == ox.as_dict() and int(ix.free_count.item()) == ofc
    n_shared = b.shared_prefix // B
    s0 = b.sharing_seqs[0]
    for s in b.sharing_seqs[1:]:
        assert np.array_equal(t1[s, :n_shared], t1[s0, :n_shared])
    # the decode step: one more token per sequence; blocks already held are kept
    nb_old = -(-lens_old.astype(np.int64) // B)
    fresh2 = pkv.paged_block_allocate(ix, keys, g["context_lens"], dev(nb_old.astype(np.int32)), B, tables)
    torch.cuda.synchronize()
    ox, ot2, ofresh2, ofc2, _ = oracle.block_allocate(ox, free_ids, ofc, keys_h, b.context_lens,
                                                       nb_old.astype(np.int32), B, ot)
    t2, f2 = tables.cpu().numpy(), fresh2.cpu().numpy()
    assert np.array_equal(t2, ot2) and np.array_equal(f2, ofresh2)
    assert int(ix.free_count.item()) == ofc2
    assert f2.sum() == int(np.sum(lens_old % B == 0))      # a new block where the old one was full
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0
    # a pool filled through the new tables; the append writes the decode tokens into it
    fresh_all = np.maximum(f1, f2)
    kn, vn = _fill_from(b, t2, fresh_all, g["k_pool"], g["v_pool"])
    pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"], g["new_starts"],
                        g["k_new"], g["v_new"])
    pkv.paged_kv_append(kn, vn, tables, g["context_lens_old"], g["new_starts"], g["k_new"], g["v_new"])
    kw = dict(max_context_len=b.max_context_len, max_q_rows_per_seq=1, sinks=g["sinks"], causal=b.causal)
    ref = pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                      g["context_lens"], **kw)
    got = pkv.paged_attention_forward(kn, vn, g["q"], g["q_starts"], tables, g["context_lens"], **kw)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(got), host_bits(ref))
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0
