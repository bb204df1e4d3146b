"""GPU keyed sampled accept against the oracle: draws, accept lengths, emitted tokens and
accepted rows bit-exact (TensorFold article, sections "先记住一条铁律" and "接受规则")."""
import numpy as np
import pytest

import oracle
from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


def _check(pkv, logits, q_starts, drafts, positions, seed, temperature, min_p=0.0, parents=None, top_k=0,
           top_p=1.0):
    got = pkv.spec_accept_sampled(dev(logits), dev(q_starts), dev(drafts), dev(positions), seed=seed,
                                  temperature=temperature, min_p=min_p, top_k=top_k, top_p=top_p,
                                  parents=None if parents is None else dev(parents))
    torch.cuda.synchronize()
    ref = oracle.spec_accept_sampled(logits, q_starts, drafts, positions, seed, temperature, min_p, parents,
                                     top_k=top_k, top_p=top_p)
    for g, r, what in zip(got, ref, ("draws", "accept_len", "out_tokens", "accepted_rows")):
        assert np.array_equal(g.cpu().numpy(), r), what
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0
    return ref


@pytest.mark.parametrize("temperature,min_p", [(1.0, 0.0), (0.7, 0.05), (1.3, 0.5), (0.0, 0.0)])
def test_chains_bit_exact(pkv, temperature, min_p):
    b = wl.make_workload("spec_verify", seed=1)
    pos = (b.context_lens[np.searchsorted(b.q_starts, np.arange(b.total_q_rows), side="right") - 1]
           + np.arange(b.total_q_rows)).astype(np.int32)
    _check(pkv, b.logits, b.q_starts, b.draft_tokens, pos, seed=1234567890123, temperature=temperature,
           min_p=min_p)


def test_trees_bit_exact(pkv):
    b = wl.make_workload("spec_tree", seed=2)
    pos = (np.arange(b.total_q_rows) * 7 + 11).astype(np.int32)
    _check(pkv, b.logits, b.q_starts, b.draft_tokens, pos, seed=99, temperature=1.0, parents=b.parents)


def test_temperature_zero_equals_greedy(pkv):
    b = wl.make_workload("spec_tree", seed=3)
    pos = np.arange(b.total_q_rows, dtype=np.int32)
    s = pkv.spec_accept_sampled(dev(b.logits), dev(b.q_starts), dev(b.draft_tokens), dev(pos), seed=5,
                                temperature=0.0, parents=dev(b.parents))
    g = pkv.spec_accept_tree_greedy(dev(b.logits), dev(b.q_starts), dev(b.draft_tokens), dev(b.parents))
    for x, y in zip(s, g):
        assert np.array_equal(x.cpu().numpy(), y.cpu().numpy())


@pytest.mark.parametrize("V", [1, 7, 1001, 32003])
def test_odd_vocabularies(pkv, V):
    rng = np.random.default_rng(V)
    lg = rng.standard_normal((9, V)).astype(np.float32)
    qs = np.array([0, 4, 9], np.int32)
    drafts = rng.integers(0, V, 9).astype(np.int32)
    pos = rng.integers(0, 1 << 20, 9).astype(np.int32)
    _check(pkv, lg, qs, drafts, pos, seed=(1 << 40) + 3, temperature=0.9, min_p=0.02)


def test_exact_ties_go_to_the_lowest_token(pkv):
    from test_oracle_sampling import colliding_tokens
    seed, pos = 7, 11
    v1, v2 = colliding_tokens(oracle, seed, pos)
    V = ((v2 + 8) // 4) * 4
    row = np.full((1, V), -100.0, np.float32)
    row[0, [v1, v2]] = 50.0
    ref = _check(pkv, row, np.array([0, 1], np.int32), np.array([-1], np.int32), np.array([pos], np.int32),
                 seed=seed, temperature=1.0)
    assert ref[0][0] == v1


@pytest.mark.parametrize("top_k,top_p,min_p,T", [(40, 1.0, 0.0, 1.0), (0, 0.9, 0.0, 1.0), (0, 0.3, 0.0, 0.6),
                                                 (50, 0.95, 0.02, 0.8), (1, 1.0, 0.0, 1.0), (0, 1e-9, 0.0, 1.0),
                                                 (0, 1e-12, 0.0, 1.0), (151935, 0.999, 0.0, 1.5)])
def test_top_k_top_p_bit_exact(pkv, top_k, top_p, min_p, T):
    # full vocabulary (151936) spec_verify rows; chains
    b = wl.make_workload("spec_verify", seed=3, num_seqs=6)
    pos = (np.arange(b.total_q_rows) * 3 + 100).astype(np.int32)
    _check(pkv, b.logits, b.q_starts, b.draft_tokens, pos, seed=77, temperature=T, min_p=min_p, top_k=top_k,
           top_p=top_p)


def test_top_p_with_ties_and_signed_zeros(pkv):
    # equal logits at the cut are ordered by token id; -0 and +0 are one logit
    rng = np.random.default_rng(4)
    V = 4099
    lg = np.round(rng.standard_normal((6, V)) * 2).astype(np.float32)   # many exact ties
    lg[:, ::7] = -0.0
    lg[:, 3::7] = 0.0
    qs = np.array([0, 2, 6], np.int32)
    drafts = rng.integers(0, V, 6).astype(np.int32)
    pos = rng.integers(0, 1 << 20, 6).astype(np.int32)
    for top_k, top_p in ((100, 1.0), (0, 0.5), (0, 0.97), (33, 0.8)):
        _check(pkv, lg, qs, drafts, pos, seed=12, temperature=1.0, top_k=top_k, top_p=top_p)


def test_top_k_top_p_trees(pkv):
    b = wl.make_workload("spec_tree", seed=5, num_seqs=4)
    pos = (np.arange(b.total_q_rows) * 5 + 3).astype(np.int32)
    _check(pkv, b.logits, b.q_starts, b.draft_tokens, pos, seed=8, temperature=1.0, parents=b.parents, top_k=20,
           top_p=0.8)
