"""Seeded synthetic inputs shaped like the serving workloads the pages describe.

This module only draws random numbers and lays out buffers: block pools, block
tables, context lengths, query rows, new K/V rows, sink logits, verify logits
and draft chains.  It holds none of the arithmetic of attention, append or
accept, so the float64 oracle and the CUDA path can both consume its output.
Everything is numpy (bf16 values are carried as their uint16 bit patterns).

Workloads (sizes from the continuous-batching / speculative-decoding pages):
  tiny_decode       4 seqs, cached lengths {37,100,203,800}, 8 q / 2 kv heads,
                    head_dim 64, block 16; append 1 token each, 1 decode row.
  ministral_decode  4 seqs, lengths U[760,840], 32 q / 8 kv heads, head_dim
                    128, block 16, 40 layers with independent pools.
  cb_mix            64 seqs, cached lengths log-uniform, 48 of them sharing a
                    2900-token prefix through the same physical full blocks,
                    40 q / 8 kv heads, head_dim 128, block 16; append 1 token
                    each, 1 decode row.
  spec_verify       16 seqs, lengths U[4096,32768] including a causal verify
                    window of U{1..16} rows whose K/V are appended first,
                    32 q / 8 kv heads, head_dim 128; verify logits over a
                    151936-token vocabulary and a draft chain per sequence.
  sinks_scale       128 seqs x 8192 tokens, 64 q / 8 kv heads, head_dim 64,
                    block 32, one fp32 sink logit per q head.
  spec_tree         spec_verify's shapes with each window a random draft tree
                    (per-row ancestor masks, parent indices, tree drafts).
  sparse_gather     cb_mix's sequences, each decode row attending over a list of
                    [its last 128 | 512 older] key positions.
  prefill_mix       16 seqs, cached lengths U[1024,8192], each appending a
                    256-token prefill chunk with causal rows, 32 q / 8 kv heads,
                    head_dim 128, block 16.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BF16_QNAN = np.uint16(0x7FC0)
_CHUNK = 1 << 22  # elements per independently seeded chunk (fixed: results do not depend on threads)


def _seed_seq(seed) -> np.random.SeedSequence:
    return seed if isinstance(seed, np.random.SeedSequence) else np.random.SeedSequence(seed)


def _workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def _round_f32_to_bf16_bits(buf: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Only finite inputs are produced here, so the integer form of the rounding is exact.
    """
    u = buf.view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb
    u >>= 16
    return u.astype(np.uint16)


def _fill_parallel(seed_seq: np.random.SeedSequence, out_flat: np.ndarray, kind: str, scale: float):
    n = out_flat.shape[0]
    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks == 0:
        return
    children = seed_seq.spawn(nchunks)

    def work(i):
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.Generator(np.random.PCG64(children[i]))
        tmp = g.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            tmp *= np.float32(scale)
        if kind == "bf16":
            out_flat[lo:hi] = _round_f32_to_bf16_bits(tmp)
        else:
            out_flat[lo:hi] = tmp

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_workers()) as ex:
            list(ex.map(work, range(nchunks)))


def normal_bf16(seed_seq: np.random.SeedSequence, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) samples rounded to bf16, as uint16 bits."""
    out = np.empty(int(np.prod(shape)), dtype=np.uint16)
    _fill_parallel(seed_seq, out, "bf16", std)
    return out.reshape(shape)


def normal_f32(seed_seq: np.random.SeedSequence, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(int(np.prod(shape)), dtype=np.float32)
    _fill_parallel(seed_seq, out, "f32", std)
    return out.reshape(shape)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 bits (nearest, ties to even)."""
    return _round_f32_to_bf16_bits(np.array(x, dtype=np.float32, copy=True))


@dataclass
class PagedBatch:
    """One batch of paged-KV work.  bf16 tensors are uint16 bit patterns.

    k_pool, v_pool: [layers, num_blocks, H_kv, block_size, head_dim]; the slots of
        the tokens that the batch appends still hold filler until the append runs.
    block_tables: int32 [S, max_blocks_per_seq]; entries past a sequence's last
        block are -1.
    context_lens_old: int32 [S] tokens cached before the append.
    context_lens: int32 [S] tokens cached after the append (what attention reads).
    new_starts: int32 [S+1] offsets of each sequence's rows in k_new / v_new.
    k_new, v_new: [layers, R_new, H_kv, head_dim] rows to append.
    q_starts: int32 [S+1]; q: [layers, R, H_q, head_dim] query rows.
    sinks: float32 [H_q] or None.
    """
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    k_pool: np.ndarray
    v_pool: np.ndarray
    block_tables: np.ndarray
    context_lens_old: np.ndarray
    context_lens: np.ndarray
    new_starts: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    q_starts: np.ndarray
    q: np.ndarray
    causal: bool
    sinks: Optional[np.ndarray] = None
    shared_block_ids: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    sharing_seqs: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    logits: Optional[np.ndarray] = None        # float32 [R, vocab] (verify workloads)
    draft_tokens: Optional[np.ndarray] = None  # int32 [R]; slot 0 of each sequence is -1
    planted_targets: Optional[np.ndarray] = None  # int32 [R]: token given the planted maximum
    parents: Optional[np.ndarray] = None       # int32 [R]: draft-tree parent node of each row (-1 at roots)
    tree_masks: Optional[np.ndarray] = None    # uint32 [R]: bit i = the row sees window token i
    shared_prefix: int = 0                     # tokens the sharing sequences have in common
    key_idx: Optional[np.ndarray] = None       # int32 [sets, R, max_keys]: per-row key positions (-1 pad)
    key_counts: Optional[np.ndarray] = None    # int32 [sets, R]

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def layers(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[1])

    @property
    def total_q_rows(self) -> int:
        return int(self.q_starts[-1])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_q_rows_per_seq(self) -> int:
        return int(np.diff(self.q_starts).max()) if self.num_seqs else 0


def build_batch(seed, *, name: str, lens: np.ndarray, n_new: np.ndarray, q_rows: np.ndarray,
                num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                causal: bool, with_sinks: bool = False, layers: int = 1,
                shared_prefix: int = 0, sharing: Optional[np.ndarray] = None,
                filler: str = "random", slack_frac: float = 0.10,
                extra_table_cols: int = 0) -> PagedBatch:
    """Lay out a paged batch.

    lens: final context length per sequence (after the append); n_new: tokens the
    batch appends per sequence (the last n_new positions); q_rows: query rows per
    sequence.  ``sharing`` marks sequences whose first ``shared_prefix`` tokens are
    the same; their full prefix blocks are one set of physical blocks, the partial
    prefix tail sits (with identical values) in each sequence's own block.
    filler: "random" puts N(0,1) values in every slot no token owns (pool slack,
    block tails, slots awaiting the append); "nan" puts bf16 NaN there instead.
    """
    root = _seed_seq(seed)
    (s_struct, s_k, s_v, s_q, s_kn, s_vn, s_sink) = root.spawn(7)
    rng = np.random.Generator(np.random.PCG64(s_struct))
    lens = np.asarray(lens, dtype=np.int64)
    n_new = np.asarray(n_new, dtype=np.int64)
    q_rows = np.asarray(q_rows, dtype=np.int64)
    S = lens.shape[0]
    B = block_size
    if sharing is None:
        sharing = np.zeros(S, dtype=bool)
    sharing = np.asarray(sharing, dtype=bool)
    old = lens - n_new
    assert np.all(old >= 0)
    n_full_shared = shared_prefix // B if sharing.any() else 0
    if sharing.any():
        assert np.all(old[sharing] >= shared_prefix), "sharing sequences must hold the whole prefix"
    nblk = (lens + B - 1) // B
    private = nblk - np.where(sharing, n_full_shared, 0)
    n_unique = int(n_full_shared + private.sum())
    slack = max(1, int(math.ceil(slack_frac * n_unique)))
    num_blocks = n_unique + slack
    perm = rng.permutation(num_blocks).astype(np.int32)
    shared_ids = perm[:n_full_shared]
    max_blocks = int(max(1, nblk.max() if S else 1)) + extra_table_cols
    tables = np.full((S, max_blocks), -1, dtype=np.int32)
    cursor = n_full_shared
    for s in range(S):
        j0 = 0
        if sharing[s]:
            tables[s, :n_full_shared] = shared_ids
            j0 = n_full_shared
        cnt = int(nblk[s] - j0)
        tables[s, j0:j0 + cnt] = perm[cursor:cursor + cnt]
        cursor += cnt
    assert cursor == n_unique

    H, D = num_kv_heads, head_dim
    shape = (layers, num_blocks, H, B, D)
    k_pool = normal_bf16(s_k, shape)
    v_pool = normal_bf16(s_v, shape)

    # identical prefix tail tokens in every sharing sequence's own partial block
    tail = shared_prefix - n_full_shared * B if sharing.any() else 0
    if tail > 0:
        idx = np.nonzero(sharing)[0]
        src_blk = tables[idx[0], n_full_shared]
        for s in idx[1:]:
            dst_blk = tables[s, n_full_shared]
            k_pool[:, dst_blk, :, :tail, :] = k_pool[:, src_blk, :, :tail, :]
            v_pool[:, dst_blk, :, :tail, :] = v_pool[:, src_blk, :, :tail, :]

    if filler == "nan":
        owned = np.zeros((num_blocks, B), dtype=bool)
        for s in range(S):
            for t0 in range(0, int(old[s]), B):
                blk = tables[s, t0 // B]
                owned[blk, : min(B, int(old[s]) - t0)] = True
        unowned = np.broadcast_to(~owned[:, None, :], (num_blocks, H, B))
        k_pool[:, unowned] = BF16_QNAN
        v_pool[:, unowned] = BF16_QNAN
    elif filler != "random":
        raise ValueError(filler)

    new_starts = np.zeros(S + 1, dtype=np.int32)
    new_starts[1:] = np.cumsum(n_new)
    q_starts = np.zeros(S + 1, dtype=np.int32)
    q_starts[1:] = np.cumsum(q_rows)
    r_new = int(new_starts[-1])
    R = int(q_starts[-1])
    k_new = normal_bf16(s_kn, (layers, r_new, H, D))
    v_new = normal_bf16(s_vn, (layers, r_new, H, D))
    q = normal_bf16(s_q, (layers, R, num_q_heads, D))
    sinks = normal_f32(s_sink, (num_q_heads,)) if with_sinks else None
    return PagedBatch(name=name, num_q_heads=num_q_heads, num_kv_heads=H, head_dim=D,
                      block_size=B, k_pool=k_pool, v_pool=v_pool, block_tables=tables,
                      context_lens_old=old.astype(np.int32), context_lens=lens.astype(np.int32),
                      new_starts=new_starts, k_new=k_new, v_new=v_new, q_starts=q_starts, q=q,
                      causal=causal, sinks=sinks, shared_block_ids=shared_ids.astype(np.int32),
                      sharing_seqs=np.nonzero(sharing)[0].astype(np.int32),
                      shared_prefix=int(shared_prefix) if sharing.any() else 0)


def add_verify_logits(batch: PagedBatch, seed, vocab: int, std: float = 2.0,
                      hit_prob: float = 0.7, planted_value: float = 20.0) -> PagedBatch:
    """Attach verify-row logits and a draft chain to ``batch``.

    Logits are N(0, std^2); one token per row (drawn uniformly) is given the value
    ``planted_value`` (10 sigma at std 2), which makes it that row's maximum.  The
    draft for row j >= 1 of a sequence is row j-1's planted token with probability
    ``hit_prob``, otherwise a uniformly drawn token (which may match by chance).
    Slot 0 of every sequence holds -1 (row 0 carries no draft).
    """
    s_logit, s_pick = _seed_seq(seed).spawn(2)
    rng = np.random.Generator(np.random.PCG64(s_pick))
    R = batch.total_q_rows
    logits = normal_f32(s_logit, (R, vocab), std)
    planted = rng.integers(0, vocab, size=R).astype(np.int32)
    logits[np.arange(R), planted] = np.float32(planted_value)
    drafts = np.full(R, -1, dtype=np.int32)
    coins = rng.random(R)
    randoms = rng.integers(0, vocab, size=R).astype(np.int32)
    for s in range(batch.num_seqs):
        r0, r1 = int(batch.q_starts[s]), int(batch.q_starts[s + 1])
        for r in range(r0 + 1, r1):
            drafts[r] = planted[r - 1] if coins[r] < hit_prob else randoms[r]
    batch.logits = logits
    batch.draft_tokens = drafts
    batch.planted_targets = planted
    return batch


def add_draft_trees(batch: PagedBatch, seed, vocab: int, std: float = 2.0, hit_prob: float = 0.7,
                    planted_value: float = 20.0) -> PagedBatch:
    """Attach draft trees to a verify batch: node j >= 1 of each sequence takes a parent
    drawn uniformly from nodes 0..j-1 and, with probability ``hit_prob``, the parent's
    planted target token as its draft (else a uniform token).  Also fills the per-row
    visibility masks (a node sees its ancestors and itself) and the verify logits (as in
    ``add_verify_logits``)."""
    s_logit, s_pick = _seed_seq(seed).spawn(2)
    rng = np.random.Generator(np.random.PCG64(s_pick))
    R = batch.total_q_rows
    logits = normal_f32(s_logit, (R, vocab), std)
    planted = rng.integers(0, vocab, size=R).astype(np.int32)
    logits[np.arange(R), planted] = np.float32(planted_value)
    parents = np.full(R, -1, dtype=np.int32)
    drafts = np.full(R, -1, dtype=np.int32)
    masks = np.zeros(R, dtype=np.uint32)
    for s in range(batch.num_seqs):
        r0, r1 = int(batch.q_starts[s]), int(batch.q_starts[s + 1])
        for j in range(r1 - r0):
            if j == 0:
                masks[r0] = 1
                continue
            par = int(rng.integers(0, j))
            parents[r0 + j] = par
            drafts[r0 + j] = planted[r0 + par] if rng.random() < hit_prob else int(rng.integers(0, vocab))
            masks[r0 + j] = masks[r0 + par] | np.uint32(1 << j)
    batch.logits = logits
    batch.draft_tokens = drafts
    batch.planted_targets = planted
    batch.parents = parents
    batch.tree_masks = masks
    return batch


def add_key_lists(batch: PagedBatch, seed, ring: int = 128, top: int = 512, sets: int = 1) -> PagedBatch:
    """Per-row key lists for the index-list gather: the row's last `ring` cached keys
    followed by `top` distinct positions drawn uniformly from the keys before them (in
    random order, as an indexer's top-k would arrive), padded with -1.  `sets`
    independent list sets let a benchmark change the lists every step."""
    rng = np.random.Generator(np.random.PCG64(_seed_seq(seed)))
    R = batch.total_q_rows
    width = ring + top
    idx = np.full((sets, R, width), -1, dtype=np.int32)
    cnt = np.zeros((sets, R), dtype=np.int32)
    row_seq = np.searchsorted(batch.q_starts, np.arange(R), side="right") - 1
    W = np.diff(batch.q_starts)
    for k in range(sets):
        for r in range(R):
            s = row_seq[r]
            # the keys row r may see: up to its own position in a causal window
            L = int(batch.context_lens[s] - W[s] + (r - batch.q_starts[s]) + 1) if batch.causal \
                else int(batch.context_lens[s])
            nr = min(ring, L)
            recent = np.arange(L - nr, L, dtype=np.int32)
            pool = L - nr
            nt = min(top, pool)
            older = rng.choice(pool, size=nt, replace=False).astype(np.int32) if nt > 0 else np.zeros(0, np.int32)
            lst = np.concatenate([recent, older])
            idx[k, r, :len(lst)] = lst
            cnt[k, r] = len(lst)
    batch.key_idx = idx
    batch.key_counts = cnt
    return batch


def _loguniform_int(rng, lo, hi, size):
    return np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), size=size))).astype(np.int64)


WORKLOADS = ("tiny_decode", "ministral_decode", "cb_mix", "spec_verify", "sinks_scale", "spec_tree",
             "sparse_gather", "prefill_mix")
VOCAB = 151936


def make_workload(name: str, seed: int = 0, filler: str = "random", layers: Optional[int] = None,
                  num_seqs: Optional[int] = None) -> PagedBatch:
    """Build one of the named workloads (see the module docstring).

    num_seqs shrinks or grows the batch of cb_mix / spec_verify / sinks_scale with the
    same per-sequence distributions (cb_mix keeps three quarters of it sharing the
    prefix); used to profile a smaller case of the same kernels."""
    base = np.random.SeedSequence([seed, WORKLOADS.index(name)])
    s_shape, s_batch, s_extra = base.spawn(3)
    rng = np.random.Generator(np.random.PCG64(s_shape))
    if name == "tiny_decode":
        old = np.array([37, 100, 203, 800])
        return build_batch(s_batch, name=name, lens=old + 1, n_new=np.ones(4, np.int64),
                           q_rows=np.ones(4, np.int64), num_q_heads=8, num_kv_heads=2,
                           head_dim=64, block_size=16, causal=False, filler=filler)
    if name == "ministral_decode":
        lens = rng.integers(760, 841, size=4)
        return build_batch(s_batch, name=name, lens=lens, n_new=np.zeros(4, np.int64),
                           q_rows=np.ones(4, np.int64), num_q_heads=32, num_kv_heads=8,
                           head_dim=128, block_size=16, causal=False, filler=filler,
                           layers=40 if layers is None else layers)
    if name == "cb_mix":
        S = num_seqs or 64
        n_share, prefix = (3 * S) // 4, 2900
        sharing = np.zeros(S, dtype=bool)
        sharing[rng.permutation(S)[:n_share]] = True
        old = np.where(sharing, _loguniform_int(rng, prefix + 1, 32767, S),
                       _loguniform_int(rng, 128, 32767, S))
        return build_batch(s_batch, name=name, lens=old + 1, n_new=np.ones(S, np.int64),
                           q_rows=np.ones(S, np.int64), num_q_heads=40, num_kv_heads=8,
                           head_dim=128, block_size=16, causal=False, filler=filler,
                           shared_prefix=prefix, sharing=sharing)
    if name == "sparse_gather":
        # cb_mix's sequences, each decode row reading [its last 128 keys | 512 older keys]
        S = num_seqs or 64
        n_share, prefix = (3 * S) // 4, 2900
        sharing = np.zeros(S, dtype=bool)
        sharing[rng.permutation(S)[:n_share]] = True
        old = np.where(sharing, _loguniform_int(rng, prefix + 1, 32767, S),
                       _loguniform_int(rng, 128, 32767, S))
        b = build_batch(s_batch, name=name, lens=old + 1, n_new=np.ones(S, np.int64),
                        q_rows=np.ones(S, np.int64), num_q_heads=40, num_kv_heads=8,
                        head_dim=128, block_size=16, causal=False, filler=filler,
                        shared_prefix=prefix, sharing=sharing)
        return add_key_lists(b, s_extra, ring=128, top=512, sets=4)
    if name == "prefill_mix":
        # chunked prefill in bounded 256-token chunks: the chunk's K/V are appended first and
        # its rows attend causally over the cached context and the chunk
        S = num_seqs or 16
        old = rng.integers(1024, 8193, size=S)
        chunk = np.full(S, 256, np.int64)
        return build_batch(s_batch, name=name, lens=old + chunk, n_new=chunk, q_rows=chunk, num_q_heads=32,
                           num_kv_heads=8, head_dim=128, block_size=16, causal=True, filler=filler)
    if name == "spec_verify":
        S = num_seqs or 16
        lens = rng.integers(4096, 32769, size=S)
        w = rng.integers(1, 17, size=S)
        b = build_batch(s_batch, name=name, lens=lens, n_new=w, q_rows=w, num_q_heads=32,
                        num_kv_heads=8, head_dim=128, block_size=16, causal=True, filler=filler)
        return add_verify_logits(b, s_extra, VOCAB)
    if name == "spec_tree":
        S = num_seqs or 16
        lens = rng.integers(4096, 32769, size=S)
        w = rng.integers(1, 17, size=S)
        b = build_batch(s_batch, name=name, lens=lens, n_new=w, q_rows=w, num_q_heads=32,
                        num_kv_heads=8, head_dim=128, block_size=16, causal=False, filler=filler)
        return add_draft_trees(b, s_extra, VOCAB)
    if name == "sinks_scale":
        S = num_seqs or 128
        return build_batch(s_batch, name=name, lens=np.full(S, 8192), n_new=np.zeros(S, np.int64),
                           q_rows=np.ones(S, np.int64), num_q_heads=64, num_kv_heads=8,
                           head_dim=64, block_size=32, causal=False, with_sinks=True, filler=filler)
    raise KeyError(name)


def record_bytes(block_size: int, head_dim: int, bits: int) -> int:
    """Size of one (block, KV head) record of a quantised pool: K codes, V codes, K and V scales."""
    return 2 * block_size * head_dim * bits // 8 + 8 * block_size


def random_records(seed, batch: PagedBatch, bits: int, layers: int = 1, filler: str = "random"):
    """A quantised pool with the batch's geometry: uint8 [layers, num_blocks, H_kv, record].

    Codes are independent draws of a rounded N(0, (Q/3)^2) clipped to [-Q, Q] (Q = 127, 7
    or 1), stored in the codec's byte encoding (8 bits: bytes of c + 128; 4 bits: two
    nibbles of c + 8 per byte; 2 bits: four bit pairs of c + 2 per byte); since every
    code is drawn alike, where a code sits in the record does not matter.  Scales are float32 uniform in [0.5, 1.5) * 3 / Q, so
    values are about N(0, 1) like the bf16 workloads.  filler "nan" stores NaN scales
    in every slot no cached token owns (pool slack, block tails, slots awaiting the
    append)."""
    s_codes, s_scales = _seed_seq(seed).spawn(2)
    B, D, H = batch.block_size, batch.head_dim, batch.num_kv_heads
    nb = batch.k_pool.shape[1] if batch.k_pool is not None else int(batch.block_tables.max()) + 1
    C = B * D * bits // 8
    rb = record_bytes(B, D, bits)
    q = (1 << (bits - 1)) - 1
    rec = np.empty((layers, nb, H, rb), dtype=np.uint8)
    codes = normal_f32(s_codes, (layers, nb, H, 2 * C * (8 // bits)), std=q / 3.0)
    codes = np.clip(np.rint(codes), -q, q).astype(np.int16)
    if bits == 8:
        rec[..., :2 * C] = (codes + 128).astype(np.uint8)
    elif bits == 4:
        nib = (codes + 8).astype(np.uint8)
        rec[..., :2 * C] = nib[..., 0::2] | (nib[..., 1::2] << 4)
    else:
        f = (codes + 2).astype(np.uint8)
        rec[..., :2 * C] = f[..., 0::4] | (f[..., 1::4] << 2) | (f[..., 2::4] << 4) | (f[..., 3::4] << 6)
    del codes
    rng = np.random.Generator(np.random.PCG64(s_scales))
    scales = ((0.5 + rng.random((layers, nb, H, 2, B))) * (3.0 / q)).astype(np.float32)
    if filler == "nan":
        owned = np.zeros((nb, B), dtype=bool)
        for sq in range(batch.num_seqs):
            old = int(batch.context_lens_old[sq])
            for t0 in range(0, old, B):
                owned[batch.block_tables[sq, t0 // B], : min(B, old - t0)] = True
        scales[:, ~owned[:, None, None, :].repeat(H, 1).repeat(2, 2)] = np.nan
    elif filler != "random":
        raise ValueError(filler)
    rec[..., 2 * C:] = scales.reshape(layers, nb, H, 2 * B).view(np.uint8).reshape(layers, nb, H, 8 * B)
    return rec


def context_token_ids(batch: PagedBatch, seed, vocab: int = VOCAB):
    """Token ids of every sequence's context, for the block-key workloads.

    Uniform ids in [0, vocab); the sharing sequences begin with the same
    batch.shared_prefix ids.  Returns (tokens int32 [sum of context_lens],
    token_starts int32 [S+1])."""
    rng = np.random.Generator(np.random.PCG64(_seed_seq(seed)))
    lens = batch.context_lens.astype(np.int64)
    starts = np.zeros(len(lens) + 1, np.int64)
    starts[1:] = np.cumsum(lens)
    tokens = rng.integers(0, vocab, size=int(starts[-1]), dtype=np.int64).astype(np.int32)
    if batch.shared_prefix and len(batch.sharing_seqs):
        prefix = rng.integers(0, vocab, size=batch.shared_prefix, dtype=np.int64).astype(np.int32)
        for s in batch.sharing_seqs:
            tokens[starts[s]:starts[s] + batch.shared_prefix] = prefix
    return tokens, starts.astype(np.int32)


def select_seqs(batch: PagedBatch, seqs) -> PagedBatch:
    """A batch holding only the listed sequences (same pool, same physical blocks).

    Used to run one sequence 'alone' against the same pool, or to cut a bounded
    sample for CPU timing.
    """
    seqs = np.asarray(seqs, dtype=np.int64)
    q_rows = np.diff(batch.q_starts)[seqs]
    n_new = np.diff(batch.new_starts)[seqs]
    q_starts = np.zeros(len(seqs) + 1, np.int32)
    q_starts[1:] = np.cumsum(q_rows)
    new_starts = np.zeros(len(seqs) + 1, np.int32)
    new_starts[1:] = np.cumsum(n_new)
    q_idx = np.concatenate([np.arange(batch.q_starts[s], batch.q_starts[s + 1]) for s in seqs]) \
        if len(seqs) else np.zeros(0, np.int64)
    n_idx = np.concatenate([np.arange(batch.new_starts[s], batch.new_starts[s + 1]) for s in seqs]) \
        if len(seqs) else np.zeros(0, np.int64)
    sub = PagedBatch(name=batch.name + "[sel]", num_q_heads=batch.num_q_heads,
                     num_kv_heads=batch.num_kv_heads, head_dim=batch.head_dim,
                     block_size=batch.block_size, k_pool=batch.k_pool, v_pool=batch.v_pool,
                     block_tables=np.ascontiguousarray(batch.block_tables[seqs]),
                     context_lens_old=batch.context_lens_old[seqs].copy(),
                     context_lens=batch.context_lens[seqs].copy(), new_starts=new_starts,
                     k_new=np.ascontiguousarray(batch.k_new[:, n_idx]),
                     v_new=np.ascontiguousarray(batch.v_new[:, n_idx]),
                     q_starts=q_starts, q=np.ascontiguousarray(batch.q[:, q_idx]),
                     causal=batch.causal, sinks=batch.sinks,
                     shared_block_ids=batch.shared_block_ids,
                     sharing_seqs=np.nonzero(np.isin(seqs, batch.sharing_seqs))[0].astype(np.int32),
                     shared_prefix=batch.shared_prefix)
    if batch.logits is not None:
        sub.logits = np.ascontiguousarray(batch.logits[q_idx])
        sub.draft_tokens = batch.draft_tokens[q_idx].copy()
        sub.planted_targets = batch.planted_targets[q_idx].copy()
    if batch.parents is not None:
        sub.parents = batch.parents[q_idx].copy()
        sub.tree_masks = batch.tree_masks[q_idx].copy()
    if batch.key_idx is not None:
        sub.key_idx = np.ascontiguousarray(batch.key_idx[:, q_idx])
        sub.key_counts = np.ascontiguousarray(batch.key_counts[:, q_idx])
    return sub
