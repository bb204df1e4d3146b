"""GPU chained block keys against the oracle, bit-exact.

TensorSharp "高级功能", section "连续批处理与分页 KV 缓存": every full block is
content-hashed so identical prefixes share blocks.  Integer work: every key must
equal the oracle's, including the zeros past each sequence's full blocks.
"""
import types

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


def _gpu(pkv, tokens, starts, B, seed, max_blocks, chain_in=None):
    ci = None if chain_in is None else dev(np.asarray(chain_in, np.uint64).view(np.int64))
    out = pkv.paged_block_hashes(dev(tokens), dev(starts), B, seed, max_blocks, chain_in=ci)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint64)


def _lens_batch(lens, sharing=(), prefix=0):
    return types.SimpleNamespace(context_lens=np.asarray(lens, np.int32),
                                 sharing_seqs=np.asarray(sharing, np.int32), shared_prefix=prefix)


def _check(pkv, tokens, starts, B, seed, max_blocks, chain_in=None):
    got = _gpu(pkv, tokens, starts, B, seed, max_blocks, chain_in)
    ref = oracle.block_hashes(tokens, starts, B, seed, max_blocks, chain_in=chain_in)
    assert np.array_equal(got, ref)
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0
    return got


@pytest.mark.parametrize("B", [16, 32, 7, 1])
def test_ragged_small(pkv, B):
    # lengths spanning several 32-block chunks, partial blocks, empty and sub-block sequences
    lens = [0, 3, B, B + 1, 33 * B + 5, 64 * B, 70 * B + B - 1, 5]
    toks, starts = wl.context_token_ids(_lens_batch(lens), seed=B, vocab=1 << 31)
    _check(pkv, toks, starts, B, 0xDEADBEEFCAFEF00D, 80)


def test_cb_mix_lengths_full_size(pkv):
    # 64 sequences, log-uniform 128..32768 tokens, 48 of them sharing a 2900-token prefix
    rng = np.random.default_rng(11)
    S, prefix = 64, 2900
    sharing = rng.permutation(S)[:48]
    lens = wl._loguniform_int(rng, 128, 32768, S)
    lens[sharing] = wl._loguniform_int(rng, prefix + 1, 32768, len(sharing))
    b = _lens_batch(lens, np.sort(sharing), prefix)
    toks, starts = wl.context_token_ids(b, seed=5)
    keys = _check(pkv, toks, starts, 16, 1234, 2048)
    full_shared = prefix // 16
    first = keys[b.sharing_seqs[0], :full_shared]
    for s in b.sharing_seqs[1:]:
        assert np.array_equal(keys[s, :full_shared], first)   # shared prefix -> same block keys


def test_continuation(pkv):
    rng = np.random.default_rng(12)
    B = 16
    lens = [40 * B + 3, 2 * B, 0, 100 * B + 9]
    toks, starts = wl.context_token_ids(_lens_batch(lens), seed=12)
    chain = rng.integers(0, 2**63, size=len(lens), dtype=np.int64).astype(np.uint64)
    _check(pkv, toks, starts, B, 0, 128, chain_in=chain)


def test_truncation_and_bad_range_flagged(pkv):
    B = 16
    toks, starts = wl.context_token_ids(_lens_batch([10 * B, 3 * B]), seed=13)
    got = _gpu(pkv, toks, starts, B, 9, 4)
    ref = oracle.block_hashes(toks[:4 * B], np.array([0, 4 * B], np.int32), B, 9, 4)
    assert np.array_equal(got[0], ref[0])                       # keys of the first 4 blocks
    rc, bits = pkv.device_status()
    assert rc == -5 and bits == 2           # PKV_DEV_TABLE_OVERRUN
    bad = np.array([0, 3 * B, 5 * B], np.int32)                 # second range past total_tokens
    got = _gpu(pkv, toks[:4 * B].copy(), bad, B, 9, 4)
    assert np.all(got[1] == 0)
    rc, bits = pkv.device_status()
    assert rc == -2 and bits == 64              # PKV_DEV_BAD_RANGE
