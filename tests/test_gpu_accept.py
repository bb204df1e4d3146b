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
