"""Pins for the oracle's keyed sampler and sampled accept (no GPU).

TensorFold article, section "先记住一条铁律": every draw is keyed by seed, absolute position and
token id, and a draft is accepted only when it equals the target's own draw; section
"接受规则": min_p (and top-k/top-p) are part of the keyed rule.  Reading: Gumbel-max over
l_v / T + g(seed, pos, v) among the tokens min_p keeps, Philox4x32-10 uniforms.
"""
import math
import os

import numpy as np
import pytest
from scipy import stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


_M0, _M1 = 0xD2511F53, 0xCD9E8D57      # Philox4x32 round multipliers (Salmon et al., SC'11)
_W0, _W1 = 0x9E3779B9, 0xBB67AE85      # key schedule (Weyl) increments


def _philox_ref(ctr, key):
    """Philox4x32-10 in plain Python integers, written from the generator's published
    definition: ten rounds of two 32x32->64 multiplies with the key bumped between rounds."""
    c = [int(x) & 0xFFFFFFFF for x in ctr]
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for rnd in range(10):
        if rnd:
            k0, k1 = (k0 + _W0) & 0xFFFFFFFF, (k1 + _W1) & 0xFFFFFFFF
        p0, p1 = _M0 * c[0], _M1 * c[2]
        c = [(p1 >> 32) ^ c[1] ^ k0, p1 & 0xFFFFFFFF, (p0 >> 32) ^ c[3] ^ k1, p0 & 0xFFFFFFFF]
    return c


def _kat_lines():
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        yield [int(x, 16) for x in line.split()]


def test_philox_known_answers(oracle_mod):
    n = 0
    for w in _kat_lines():
        assert oracle_mod.philox4x32_10(w[0:4], w[4:6]).tolist() == w[6:10]
        assert _philox_ref(w[0:4], w[4:6]) == w[6:10]      # the test's own generator, same answers
        n += 1
    assert n == 3


# (seed, position, token) cases for the counter layout: tokens 0-3 share counter 0 and
# take words 0-3; token 4 starts counter 1; large positions, ids and 64-bit seeds reach
# the high counter and key words.
_KEYED_CASES = [(0, 0, v) for v in range(9)] + [
    (0x243F6A8885A308D3, 123456, 151935), (0xFFFFFFFFFFFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF),
    (1, 2, 3), (7, 11, 4097), (0x13198A2E03707344, 99, 77), (42, 0, 151932)]


@pytest.mark.parametrize("seed,pos,v", _KEYED_CASES)
def test_keyed_uniform_counter_layout(oracle_mod, seed, pos, v):
    """The draw of token v at position pos under seed is the top 23 bits of word v mod 4 of
    Philox4x32-10 with counter (v / 4, pos, 0x6b657964, 0) and key (seed low, seed high)
    (one generator call keys four consecutive tokens).  The expected word comes from the
    test's own Philox, which the published known answers pin; swapping the word index or
    the counter packing in the oracle fails here."""
    words = _philox_ref([v >> 2, pos, 0x6B657964, 0], [seed & 0xFFFFFFFF, seed >> 32])
    code = words[v & 3] >> 9
    assert oracle_mod.keyed_uniform_bits(seed, pos, v) == code
    # the Gumbel noise built on it: g = -log(-log(u)), u = (code + 1/2) / 2^23
    u = (code + 0.5) / 2.0 ** 23
    g_ref = -math.log(-math.log(u))
    g = oracle_mod.keyed_gumbel(seed, pos, v)
    assert abs(g - g_ref) <= 2e-6 * max(1.0, abs(g_ref)), (g, g_ref)


def test_keyed_uniform_words_of_one_call_are_distinct_tokens(oracle_mod):
    """Tokens 4c .. 4c+3 read the four different words of one generator call."""
    for seed, pos in ((0, 0), (5, 1000)):
        for c in range(4):
            words = _philox_ref([c, pos, 0x6B657964, 0], [seed, 0])
            got = [oracle_mod.keyed_uniform_bits(seed, pos, 4 * c + j) for j in range(4)]
            assert got == [w >> 9 for w in words]


def test_keyed_log_accuracy(oracle_mod):
    rng = np.random.default_rng(0)
    xs = np.concatenate([np.exp(rng.uniform(-87, 88, 4000)), rng.uniform(0.5, 2.0, 2000),
                         [1.0, 2.0, 0.5, 1.5e-45, 1e-40, 3.4e38, 1.0000001, 0.99999994]]).astype(np.float32)
    for x in xs:
        got = float(oracle_mod.keyed_log(x))
        ref = math.log(float(x))
        ulp = float(np.spacing(np.float32(abs(ref)))) if ref != 0 else 1e-45
        assert abs(got - ref) <= max(4 * ulp, 1.5e-7), (x, got, ref)
    assert float(oracle_mod.keyed_log(np.float32(1.0))) == 0.0


def _one_chain(V, rows, seed=0):
    rng = np.random.default_rng(seed)
    lg = (rng.standard_normal((rows, V)) * 2).astype(np.float32)
    qs = np.array([0, rows], np.int32)
    return lg, qs


def test_zero_temperature_is_greedy(oracle_mod):
    from paged_kv_attention_forward_gb300 import workloads as wl
    b = wl.make_workload("spec_tree", seed=1)
    pos = np.arange(b.total_q_rows, dtype=np.int32) + 1000
    s = oracle_mod.spec_accept_sampled(b.logits, b.q_starts, b.draft_tokens, pos, seed=5, temperature=0.0,
                                       parents=b.parents)
    g = oracle_mod.spec_accept_tree_greedy(b.logits, b.q_starts, b.draft_tokens, b.parents)
    for x, y in zip(s, g):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("temperature", [1.0, 0.5])
def test_draws_follow_softmax(oracle_mod, temperature):
    V, R = 6, 60000
    row = np.array([1.0, 0.3, -0.5, 2.0, 0.0, -2.0], np.float32)
    lg = np.tile(row, (R, 1))
    qs = np.array([0] + list(range(1, R + 1)), np.int32)      # R one-row sequences
    pos = np.arange(R, dtype=np.int32)
    draws = oracle_mod.spec_accept_sampled(lg, qs, np.full(R, -1, np.int32), pos, seed=42,
                                           temperature=temperature)[0]
    counts = np.bincount(draws, minlength=V)
    p = np.exp(row.astype(np.float64) / temperature)
    p /= p.sum()
    chi2, pval = stats.chisquare(counts, R * p)
    assert pval > 1e-3, (counts, R * p)


def test_min_p_filter(oracle_mod):
    V, R = 5, 20000
    row = np.array([2.0, 1.9, 0.0, -1.0, 1.0], np.float32)   # probs relative to max: 1, .905, .135, .05, .368
    lg = np.tile(row, (R, 1))
    qs = np.array([0] + list(range(1, R + 1)), np.int32)
    pos = np.arange(R, dtype=np.int32)
    d = oracle_mod.spec_accept_sampled(lg, qs, np.full(R, -1, np.int32), pos, seed=3, temperature=1.0,
                                       min_p=0.3)[0]
    assert set(np.unique(d).tolist()) == {0, 1, 4}            # tokens below 0.3 x p_max never drawn
    kept = np.exp(row[[0, 1, 4]].astype(np.float64))
    chi2, pval = stats.chisquare(np.bincount(d, minlength=5)[[0, 1, 4]], R * kept / kept.sum())
    assert pval > 1e-3
    d1 = oracle_mod.spec_accept_sampled(lg[:500], qs[:501], np.full(500, -1, np.int32), pos[:500], seed=3,
                                        temperature=1.0, min_p=1.0)[0]
    assert np.all(d1 == 0)


def test_draws_are_keyed_by_seed_position_and_token(oracle_mod):
    lg, _ = _one_chain(50, 300, seed=4)
    R = lg.shape[0]
    qs = np.arange(R + 1, dtype=np.int32)
    pos = np.random.default_rng(1).permutation(10000)[:R].astype(np.int32)
    none = np.full(R, -1, np.int32)
    a = oracle_mod.spec_accept_sampled(lg, qs, none, pos, seed=9, temperature=1.0)[0]
    perm = np.random.default_rng(2).permutation(R)
    b = oracle_mod.spec_accept_sampled(lg[perm], qs, none, pos[perm], seed=9, temperature=1.0)[0]
    assert np.array_equal(a[perm], b)                          # batch order does not matter
    c = oracle_mod.spec_accept_sampled(lg, qs, none, pos, seed=10, temperature=1.0)[0]
    assert (a != c).mean() > 0.5                               # another seed, other draws
    d = oracle_mod.spec_accept_sampled(lg, qs, none, pos + 1, seed=9, temperature=1.0)[0]
    assert (a != d).mean() > 0.5                               # another position, other draws


def test_sampled_walk_accepts_exactly_the_matching_prefix(oracle_mod):
    lg, qs = _one_chain(40, 9, seed=6)
    pos = np.arange(9, dtype=np.int32) + 77
    draws = oracle_mod.spec_accept_sampled(lg, qs, np.full(9, -1, np.int32), pos, seed=1, temperature=0.8)[0]
    drafts = np.concatenate([[-1], draws[:-1]]).astype(np.int32)    # a perfect drafter
    s, n, out, rows = oracle_mod.spec_accept_sampled(lg, qs, drafts, pos, seed=1, temperature=0.8)
    assert n[0] == 8 and out.tolist() == draws.tolist() and rows[:8].tolist() == list(range(1, 9))
    drafts[5] = (draws[4] + 1) % 40                                   # first miss at node 5
    s, n, out, rows = oracle_mod.spec_accept_sampled(lg, qs, drafts, pos, seed=1, temperature=0.8)
    assert n[0] == 4 and out[:5].tolist() == draws[:5].tolist() and np.all(out[5:] == -1)


def colliding_tokens(oracle_mod, seed, pos, limit=30000):
    """Two token ids whose keyed uniform codes (as the oracle draws them) coincide."""
    seen = {}
    for v in range(limit):
        u = oracle_mod.keyed_uniform_bits(seed, pos, v)
        if u in seen:
            return seen[u], v
        seen[u] = v
    raise AssertionError("no collision found")


def test_exact_score_ties_go_to_the_lowest_token(oracle_mod):
    seed, pos = 7, 11
    v1, v2 = colliding_tokens(oracle_mod, seed, pos)
    row = np.full((1, v2 + 5), -100.0, np.float32)
    row[0, [v1, v2]] = 50.0                        # equal logits and equal noise: an exact tie
    d = oracle_mod.spec_accept_sampled(row, np.array([0, 1], np.int32), np.array([-1], np.int32),
                                       np.array([pos], np.int32), seed=seed, temperature=1.0)[0]
    assert d[0] == v1 < v2


# ------------------------------------------------------------- top-k / top-p --
def test_keyed_exp2_accuracy_and_exact_points(oracle_mod):
    import math
    ys = np.concatenate([np.linspace(-32, 0, 4001), -np.random.default_rng(3).random(2000) * 32])
    for y in ys.astype(np.float32):
        got = oracle_mod.keyed_exp2(float(y))
        ref = 2.0 ** float(y)
        assert abs(got - ref) <= 4e-7 * ref, (float(y), got, ref)
    for k in range(33):                      # integers: the polynomial is 1 at f = 0, scaling is exact
        assert oracle_mod.keyed_exp2(-float(k)) == 2.0 ** -k
    assert oracle_mod.keyed_exp2(0.0) == 1.0
    assert oracle_mod.keyed_exp2(-32.5) == 0.0 and oracle_mod.keyed_exp2(float("-inf")) == 0.0


def _weights(oracle_mod, row, T):
    """Integer weights of a row, from the oracle's exp2 and numpy float32 arithmetic."""
    r = np.asarray(row, np.float32)
    lmax = r.max()
    y = ((r - lmax) / np.float32(T)) * np.float32(1.4426950408889634)
    return [int(np.float32(oracle_mod.keyed_exp2(float(v))) * np.float32(2.0 ** 32)) for v in y.astype(np.float32)]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_topkp_kept_is_the_defined_prefix(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    V = 500
    row = (rng.standard_normal(V) * 2).astype(np.float32)
    row[rng.integers(0, V, 40)] = row[7]                  # ties, broken by token id
    T = 0.8
    n, order = oracle_mod.topkp_kept(row, T)
    assert n == V
    ref_order = np.lexsort((np.arange(V), -row.astype(np.float64)))
    assert np.array_equal(order, ref_order)
    assert oracle_mod.topkp_kept(row, T, top_k=17)[0] == 17
    W = _weights(oracle_mod, row, T)
    total = sum(W)
    for p in (0.05, 0.3, 0.5, 0.9, 0.99):
        n, _ = oracle_mod.topkp_kept(row, T, top_p=p)
        p_fix = int(np.float32(p) * np.float32(2.0 ** 32))
        thr = -(-(p_fix * total) // 2 ** 32)              # ceil, exact integers
        cum = np.cumsum([W[i] for i in ref_order], dtype=object)
        assert cum[n - 1] >= thr and (n == 1 or cum[n - 2] < thr), (p, n)
        assert oracle_mod.topkp_kept(row, T, top_k=n + 5, top_p=p)[0] == n
        assert oracle_mod.topkp_kept(row, T, top_k=max(1, n - 3), top_p=p)[0] == max(1, n - 3)
    assert oracle_mod.topkp_kept(row, T, top_p=1e-9)[0] == 1
    assert oracle_mod.topkp_kept(row, T, top_p=1.0)[0] == V


def test_topkp_draws(oracle_mod):
    rng = np.random.default_rng(9)
    V, R = 300, 400
    logits = np.tile((rng.standard_normal(V) * 1.5).astype(np.float32), (R, 1))
    qs = np.arange(R + 1, dtype=np.int32)
    drafts = np.full(R, -1, np.int32)
    pos = np.arange(R, dtype=np.int32) + 1000
    amax = int(np.argmax(logits[0]))
    # top-k 1 and a vanishing top-p leave only the argmax, whatever the noise
    s1, *_ = oracle_mod.spec_accept_sampled(logits, qs, drafts, pos, seed=5, temperature=1.0, top_k=1)
    s2, *_ = oracle_mod.spec_accept_sampled(logits, qs, drafts, pos, seed=5, temperature=1.0, top_p=1e-9)
    assert np.all(s1 == amax) and np.all(s2 == amax)
    # top-k 6: every draw is among the 6 largest; all 6 are drawn; frequencies follow the
    # renormalised softmax of those 6 (loose statistical check)
    s3, *_ = oracle_mod.spec_accept_sampled(logits, qs, drafts, pos, seed=5, temperature=1.0, top_k=6)
    top6 = np.argsort(-logits[0].astype(np.float64), kind="stable")[:6]
    assert set(s3.tolist()) <= set(top6.tolist()) and len(set(s3.tolist())) == 6
    pr = np.exp(logits[0][top6].astype(np.float64))
    pr /= pr.sum()
    cnt = np.array([np.sum(s3 == t) for t in top6])
    assert np.all(np.abs(cnt / R - pr) < 5 * np.sqrt(pr * (1 - pr) / R) + 0.01)
    # top-p keeps the prefix the kept-set function names
    n, order = oracle_mod.topkp_kept(logits[0], 1.0, top_p=0.6)
    s4, *_ = oracle_mod.spec_accept_sampled(logits, qs, drafts, pos, seed=6, temperature=1.0, top_p=0.6)
    assert set(s4.tolist()) <= set(order[:n].tolist())
    # no filter: the same draws as before the filters existed
    s5, *_ = oracle_mod.spec_accept_sampled(logits, qs, drafts, pos, seed=5, temperature=1.0)
    s6, *_ = oracle_mod.spec_accept_sampled(logits, qs, drafts, pos, seed=5, temperature=1.0, top_k=V, top_p=1.0)
    assert np.array_equal(s5, s6)


def test_topp_threshold_is_a_ceiling(oracle_mod):
    # exact integers: the threshold rounds p_fix * total / 2^32 up, never down
    rng = np.random.default_rng(11)
    assert oracle_mod.topp_threshold(1 << 31, 3) == 2            # 1.5 -> 2
    assert oracle_mod.topp_threshold(1 << 31, 4) == 2            # 2 exactly
    assert oracle_mod.topp_threshold(1, 1) == 1                  # 2^-32 -> 1
    assert oracle_mod.topp_threshold(0, 12345) == 0
    for _ in range(2000):
        p_fix = int(rng.integers(0, 1 << 32))
        total = int(rng.integers(1 << 32, 1 << 50))
        x = p_fix * total
        assert oracle_mod.topp_threshold(p_fix, total) == -(-x // (1 << 32))
