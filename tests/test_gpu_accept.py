"""GPU greedy accept against the oracle: argmax, accept lengths and emitted tokens bit-exact.

TensorFold article, section "接受规则：GPU 上的 accept 内核" (walk the draft chain to the
first child that differs from the target's choice); ties go to the lowest token id.
"""
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


def _run(pkv, logits, q_starts, drafts):
    a, n, out = pkv.spec_accept_greedy(dev(logits), dev(q_starts), dev(drafts))
    torch.cuda.synchronize()
    return a.cpu().numpy(), n.cpu().numpy(), out.cpu().numpy()


def _check(pkv, logits, q_starts, drafts):
    got = _run(pkv, logits, q_starts, drafts)
    ref = oracle.spec_accept_greedy(logits, q_starts, drafts)
    for g, r, what in zip(got, ref, ("argmax", "accept_len", "out_tokens")):
        assert np.array_equal(g, r), what
    return got


@pytest.mark.parametrize("seed", [0, 1])
def test_spec_verify_accept_bit_exact(pkv, seed):
    b = wl.make_workload("spec_verify", seed=seed)
    _, n, _ = _check(pkv, b.logits, b.q_starts, b.draft_tokens)
    assert n.max() > 0


def test_ties_across_slices_and_all_equal_rows(pkv):
    V = 151936
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((5, V)).astype(np.float32)
    lg[0, [150000, 9000, 70001]] = 30.0      # maxima in different slices: lowest index wins
    lg[1, :] = 0.5                           # all equal
    lg[2, :] = -np.inf                       # all -inf
    lg[3, [V - 1]] = 40.0                    # last element
    lg[4, [0, 1, 2, 3]] = 41.0
    qs = np.array([0, 5], np.int32)
    drafts = np.array([-1, 9000, 0, 0, V - 1], np.int32)
    a, n, out = _check(pkv, lg, qs, drafts)
    assert a.tolist() == [9000, 0, 0, V - 1, 0] and n[0] == 4


@pytest.mark.parametrize("V", [1, 3, 1001, 8193, 32000])
def test_odd_vocab_sizes(pkv, V):
    rng = np.random.default_rng(V)
    lg = rng.integers(-3, 4, size=(7, V)).astype(np.float32)    # many ties
    qs = np.array([0, 3, 7], np.int32)
    drafts = rng.integers(0, V, size=7).astype(np.int32)
    _check(pkv, lg, qs, drafts)


def test_long_windows_empty_sequences_and_batch_invariance(pkv):
    rng = np.random.default_rng(5)
    V = 4096
    W = [70, 0, 1, 33, 0, 16]
    qs = np.concatenate([[0], np.cumsum(W)]).astype(np.int32)
    R = int(qs[-1])
    lg = rng.standard_normal((R, V)).astype(np.float32)
    targets = rng.integers(0, V, size=R)
    lg[np.arange(R), targets] = 10.0
    drafts = np.full(R, -1, np.int32)
    for s in range(len(W)):
        for j in range(qs[s] + 1, qs[s + 1]):
            drafts[j] = targets[j - 1] if rng.random() < 0.97 else rng.integers(0, V)
    a, n, out = _check(pkv, lg, qs, drafts)
    assert n[1] == -1 and n[4] == -1
    for s in range(len(W)):
        r0, r1 = qs[s], qs[s + 1]
        one = _run(pkv, lg[r0:r1].copy() if r1 > r0 else np.zeros((0, V), np.float32),
                   np.array([0, r1 - r0], np.int32), drafts[r0:r1].copy())
        assert one[1][0] == n[s]
        assert np.array_equal(one[0], a[r0:r1]) and np.array_equal(one[2], out[r0:r1])


def _slice_bounds(V):
    """Every first slice boundary the argmax pass can use: the pass cuts a row into n
    slices of ceil(V / n) values rounded up to a multiple of 4, n from 1 to ceil(V / 8192)."""
    out = set()
    for n in range(2, (V + 8191) // 8192 + 1):
        c = -(-V // n)
        c = (c + 3) & ~3
        if c < V:
            out.add(c)
    return sorted(out)


@pytest.mark.parametrize("seed", [0, 1])
def test_spec_verify_accept_on_unplanted_logits(pkv, seed):
    """The speculative-verify config as stated: logits N(0, 2^2) over V = 151936 with no
    planted maximum, so a row's largest value sits only a few tenths above its runner-up,
    often in another slice of the argmax pass.  Drafts follow the config's chain rule with
    the target argmax taken from the oracle: d_j = argmax(row j-1) with probability 0.7,
    else a uniform token.  Some rows get their own two largest values moved (a permutation
    of the row, so its values keep their distribution) onto the two sides of a slice
    boundary, in both orders, and one row a copy of its maximum across a boundary (an exact
    tie: the lower index wins).  Argmax, accept lengths and emitted tokens bit-exact."""
    V = 151936
    rng = np.random.default_rng(100 + seed)
    W = rng.integers(1, 17, size=16)                       # 16 sequences, windows U{1..16}
    q_starts = np.concatenate([[0], np.cumsum(W)]).astype(np.int32)
    R = int(q_starts[-1])
    lg = (rng.standard_normal((R, V)) * 2.0).astype(np.float32)
    bounds = _slice_bounds(V)
    r = 0
    for c in bounds:
        for later_is_max in (True, False):
            if r >= R:
                break
            row = lg[r]
            top2 = np.argsort(row)[-2:]                    # runner-up, max
            hi, lo = row[top2[1]], row[top2[0]]
            pos_max, pos_2nd = (c, c - 1) if later_is_max else (c - 1, c)
            # move the two values there; what sat at the boundary takes their old places
            row_new = row.copy()
            others = [p for p in (top2[0], top2[1]) if p not in (pos_max, pos_2nd)]
            displaced = [row[p] for p in (pos_max, pos_2nd) if p not in (top2[0], top2[1])]
            for p, v in zip(others, displaced):
                row_new[p] = v
            row_new[pos_max], row_new[pos_2nd] = hi, lo
            assert sorted(row_new.tolist()) == sorted(row.tolist())
            lg[r] = row_new
            r += 1
    if r < R:                                              # an exact tie across the first boundary
        c = bounds[len(bounds) // 2]
        lg[r, c] = lg[r].max()
        lg[r, c - 1] = lg[r, c]
        r += 1
    assert r > 10
    target = oracle.argmax_rows(lg)
    drafts = np.full(R, -1, np.int32)
    coins = rng.random(R)
    randoms = rng.integers(0, V, size=R)
    for s in range(len(W)):
        for j in range(int(q_starts[s]) + 1, int(q_starts[s + 1])):
            drafts[j] = target[j - 1] if coins[j] < 0.7 else randoms[j]
    a, n, _ = _check(pkv, lg, q_starts, drafts)
    assert np.array_equal(a, target)
    assert n.max() > 0
