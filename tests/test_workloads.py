"""The seeded generators: determinism and the structure each workload promises (no GPU)."""
import numpy as np
import pytest

from paged_kv_attention_forward_gb300 import workloads as wl


@pytest.mark.parametrize("name", ["tiny_decode", "cb_mix", "spec_verify"])
def test_same_seed_same_bytes(name):
    a = wl.make_workload(name, seed=5)
    b = wl.make_workload(name, seed=5)
    for f in ("k_pool", "v_pool", "block_tables", "context_lens", "q", "k_new", "v_new"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    c = wl.make_workload(name, seed=6)
    assert not np.array_equal(a.q, c.q)


@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_tables_address_distinct_private_blocks(name):
    b = wl.make_workload(name, seed=1, layers=1)
    B = b.block_size
    owners = {}
    shared = set(b.shared_block_ids.tolist())
    for s in range(b.num_seqs):
        nblk = (int(b.context_lens[s]) + B - 1) // B
        row = b.block_tables[s]
        assert np.all(row[:nblk] >= 0) and np.all(row[:nblk] < b.num_blocks)
        assert np.all(row[nblk:] == -1)
        for j, blk in enumerate(row[:nblk].tolist()):
            if blk in shared:
                assert j < len(b.shared_block_ids) and s in b.sharing_seqs
                continue
            assert blk not in owners, "private block used twice"
            owners[blk] = s
    assert b.num_blocks > len(owners) + len(shared)        # slack blocks exist


def test_cb_mix_shape_and_shared_prefix():
    b = wl.make_workload("cb_mix", seed=0)
    assert b.num_seqs == 64 and len(b.sharing_seqs) == 48
    assert len(b.shared_block_ids) == 2900 // 16
    old = b.context_lens_old
    assert old.min() >= 128 and old.max() <= 32767
    assert np.all(old[b.sharing_seqs] >= 2901)
    assert np.array_equal(b.context_lens, old + 1)
    # the 4 prefix tokens past the last full shared block hold the same values everywhere
    nsh = len(b.shared_block_ids)
    blocks = b.block_tables[b.sharing_seqs, nsh]
    ref = b.k_pool[0, blocks[0], :, :4]
    for blk in blocks[1:]:
        assert np.array_equal(b.k_pool[0, blk, :, :4], ref)
    assert (b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size) == (40, 8, 128, 16)


def test_spec_verify_drafts_and_windows():
    b = wl.make_workload("spec_verify", seed=0)
    w = np.diff(b.q_starts)
    assert w.min() >= 1 and w.max() <= 16 and b.causal
    assert np.array_equal(np.diff(b.new_starts), w)
    assert b.logits.shape == (b.total_q_rows, wl.VOCAB)
    hits = []
    for s in range(b.num_seqs):
        r0, r1 = b.q_starts[s], b.q_starts[s + 1]
        assert b.draft_tokens[r0] == -1
        hits += [b.draft_tokens[r] == b.planted_targets[r - 1] for r in range(r0 + 1, r1)]
    assert 0.5 < np.mean(hits) < 0.9


def test_nan_filler_only_in_unowned_slots():
    b = wl.make_workload("tiny_decode", seed=0, filler="nan")
    nan = b.k_pool[0] == wl.BF16_QNAN
    B = b.block_size
    for s in range(b.num_seqs):
        for t in range(int(b.context_lens_old[s])):
            assert not nan[b.block_tables[s, t // B], :, t % B].any()
        p = int(b.context_lens_old[s])                      # slot awaiting the append
        assert nan[b.block_tables[s, p // B], :, p % B].all()


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3, 65504.0], np.float32)
    bits = wl.f32_to_bf16_bits(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6: even mantissa (1 + 2^-6) wins
    assert bits[0] == 0x3F80 and bits[1] == 0x3F80 and bits[2] == 0x3F82
    back = wl.bf16_bits_to_f32(bits)
    assert back[3] == -2.5
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -8)
