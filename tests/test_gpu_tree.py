"""GPU tree verify: attention with per-row ancestor masks and greedy accept over draft trees,
against the oracle (TensorFold article, section "接受规则：GPU 上的 accept 内核")."""
import numpy as np
import pytest

import oracle
from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import assert_close_to_oracle, dev, dev_bf16, gpu_batch, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


def _status_ok(pkv):
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0, f"device status {rc}, bits {bits:#x}"


def _tree_step(pkv, b, g=None, tree_masks=None):
    g = g or gpu_batch(b)
    pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"], g["new_starts"],
                        g["k_new"], g["v_new"])
    masks = b.tree_masks if tree_masks is None else tree_masks
    out = pkv.paged_tree_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                           g["context_lens"], dev(masks.view(np.int32)),
                                           max_context_len=b.max_context_len,
                                           max_q_rows_per_seq=b.max_q_rows_per_seq)
    torch.cuda.synchronize()
    return g, out


@pytest.mark.parametrize("seed", [0, 1])
def test_tree_attention_matches_oracle(pkv, seed):
    b = wl.make_workload("spec_tree", seed=seed)
    _, out = _tree_step(pkv, b)
    k, v = b.k_pool[0].copy(), b.v_pool[0].copy()
    oracle.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts, b.k_new[0], b.v_new[0])
    ref = oracle.paged_attention(k, v, b.q[0], b.q_starts, b.block_tables, b.context_lens,
                                 tree_masks=b.tree_masks)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, what=f"tree {seed}")
    _status_ok(pkv)


def test_chain_masks_bit_identical_to_causal_window(pkv):
    b = wl.make_workload("spec_verify", seed=4)
    chain = np.concatenate([(1 << (np.arange(w) + 1)) - 1 for w in np.diff(b.q_starts)]).astype(np.uint32)
    g, tree_out = _tree_step(pkv, b, tree_masks=chain)
    causal = pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                         g["context_lens"], max_context_len=b.max_context_len,
                                         max_q_rows_per_seq=b.max_q_rows_per_seq, causal=True)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(tree_out), host_bits(causal))


def test_tree_batch_vs_solo_bit_identical(pkv):
    b = wl.make_workload("spec_tree", seed=5)
    g, out = _tree_step(pkv, b)
    full = host_bits(out)
    for s in range(b.num_seqs):
        sub = wl.select_seqs(b, [s])
        one = pkv.paged_tree_attention_forward(
            g["k_pool"], g["v_pool"], dev_bf16(sub.q[0]), dev(sub.q_starts), dev(sub.block_tables),
            dev(sub.context_lens), dev(sub.tree_masks.view(np.int32)), max_context_len=sub.max_context_len,
            max_q_rows_per_seq=sub.max_q_rows_per_seq)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(one), full[b.q_starts[s]:b.q_starts[s + 1]]), f"seq {s}"


@pytest.mark.parametrize("seed", [0, 2])
def test_tree_accept_bit_exact(pkv, seed):
    b = wl.make_workload("spec_tree", seed=seed)
    got = pkv.spec_accept_tree_greedy(dev(b.logits), dev(b.q_starts), dev(b.draft_tokens), dev(b.parents))
    ref = oracle.spec_accept_tree_greedy(b.logits, b.q_starts, b.draft_tokens, b.parents)
    for x, y, what in zip(got, ref, ("argmax", "accept_len", "out_tokens", "accepted_rows")):
        assert np.array_equal(x.cpu().numpy(), y), what
    assert ref[1].max() > 0
    _status_ok(pkv)


def test_tree_accept_on_chains_equals_chain_accept(pkv):
    b = wl.make_workload("spec_verify", seed=6)
    parents = np.concatenate([np.arange(-1, w - 1) for w in np.diff(b.q_starts)]).astype(np.int32)
    t = pkv.spec_accept_tree_greedy(dev(b.logits), dev(b.q_starts), dev(b.draft_tokens), dev(parents))
    c = pkv.spec_accept_greedy(dev(b.logits), dev(b.q_starts), dev(b.draft_tokens))
    for x, y in zip(t[:3], c):
        assert np.array_equal(x.cpu().numpy(), y.cpu().numpy())


def test_wide_trees_and_bad_parents(pkv):
    rng = np.random.default_rng(9)
    W = [40, 1, 0, 70]                                   # more nodes than one ballot covers
    qs = np.concatenate([[0], np.cumsum(W)]).astype(np.int32)
    R, V = int(qs[-1]), 3000
    lg = rng.standard_normal((R, V)).astype(np.float32)
    tgt = rng.integers(0, V, R)
    lg[np.arange(R), tgt] = 9.0
    parents = np.full(R, -1, np.int32)
    drafts = np.full(R, -1, np.int32)
    for s in range(len(W)):
        for j in range(1, W[s]):
            parents[qs[s] + j] = max(0, j - 1 - int(rng.integers(0, 2)))
            drafts[qs[s] + j] = tgt[qs[s] + parents[qs[s] + j]] if rng.random() < 0.9 else 0
    got = pkv.spec_accept_tree_greedy(dev(lg), dev(qs), dev(drafts), dev(parents))
    ref = oracle.spec_accept_tree_greedy(lg, qs, drafts, parents)
    for x, y in zip(got, ref):
        assert np.array_equal(x.cpu().numpy(), y)
    _status_ok(pkv)
    bad = parents.copy()
    bad[qs[3] + 5] = 7                                  # parent after its child
    got = pkv.spec_accept_tree_greedy(dev(lg), dev(qs), dev(drafts), dev(bad))
    torch.cuda.synchronize()
    assert got[1].cpu().numpy()[3] == -1
    rc, bits = pkv.device_status()
    assert rc == -2 and bits & 32
