"""Float64 CPU oracle for paged-KV attention, paged K/V append and greedy accept.

TEST INFRASTRUCTURE ONLY.  This package states, plainly and slowly, what the GPU
path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
and reference arms of ``bench.py`` may import it.  The CUDA library and its
Python binding never import, link or call it, and it never imports them.

The arithmetic lives in ``pkv_oracle.c`` (plain C99, float64, OpenMP over
(sequence, KV head)); this module compiles it with gcc on first use and wraps it
with numpy.  The passages each function follows are cited in the C source:
TensorSharp "advanced features" (sections on continuous batching and the paged
KV cache, native paged attention with the sinks variant, and ForwardBatch's
paged K/V scatter) and the TensorFold article (section on the GPU accept
kernel).

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
against closed forms, invariants, library routines (torch's float64 scaled
dot-product attention, numpy's argmax) and hand-worked fixtures in
``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile pkv_oracle.c into a shared library with gcc; returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC",
               "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.oracle_paged_kv_append.argtypes = [P, P, i32, i32, i32, i32, P, i32, P, P, P, P, i32]
            lib.oracle_paged_kv_append.restype = ctypes.c_int
            lib.oracle_paged_attention.argtypes = [P, P, i32, i32, i32, i32, P, P, P, i32, P, i32,
                                                   i32, P, P, i32, P, ctypes.c_double, P, i32]
            lib.oracle_paged_attention.restype = ctypes.c_int
            lib.oracle_argmax_rows.argtypes = [P, ctypes.c_int64, i32, P]
            lib.oracle_argmax_rows.restype = None
            lib.oracle_spec_accept_greedy.argtypes = [P, i32, P, P, i32, P, P, P]
            lib.oracle_spec_accept_greedy.restype = None
            lib.oracle_spec_accept_tree_greedy.argtypes = [P, i32, P, P, P, i32, P, P, P, P]
            lib.oracle_spec_accept_tree_greedy.restype = ctypes.c_int
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_keyed_log.argtypes = [ctypes.c_float]
            lib.oracle_keyed_log.restype = ctypes.c_float
            lib.oracle_keyed_uniform_bits.argtypes = [ctypes.c_uint64, i32, i32]
            lib.oracle_keyed_uniform_bits.restype = ctypes.c_uint32
            lib.oracle_keyed_gumbel.argtypes = [ctypes.c_uint64, i32, i32]
            lib.oracle_keyed_gumbel.restype = ctypes.c_float
            lib.oracle_spec_accept_sampled.argtypes = [P, i32, P, P, P, P, ctypes.c_uint64, ctypes.c_float,
                                                       i32, ctypes.c_float, ctypes.c_float, i32, P, P, P, P]
            lib.oracle_paged_attention_sparse.argtypes = [P, P, i32, i32, i32, i32, P, P, P, i32, P, i32, P, P,
                                                          i32, i32, P, P, ctypes.c_double, P]
            lib.oracle_paged_attention_sparse.restype = ctypes.c_int
            lib.oracle_topp_threshold.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.oracle_topp_threshold.restype = ctypes.c_uint64
            lib.oracle_keyed_exp2.argtypes = [ctypes.c_float]
            lib.oracle_keyed_exp2.restype = ctypes.c_float
            lib.oracle_topkp_kept.argtypes = [P, i32, ctypes.c_float, i32, ctypes.c_float, P]
            lib.oracle_topkp_kept.restype = i32
            lib.oracle_spec_accept_sampled.restype = ctypes.c_int
            lib.oracle_fnv1a64.argtypes = [P, ctypes.c_int64]
            lib.oracle_fnv1a64.restype = ctypes.c_uint64
            lib.oracle_splitmix64_mix.argtypes = [ctypes.c_uint64]
            lib.oracle_splitmix64_mix.restype = ctypes.c_uint64
            lib.oracle_block_hashes.argtypes = [P, P, i32, i32, ctypes.c_uint64, P, P, i32]
            lib.oracle_block_hashes.restype = ctypes.c_int
            lib.oracle_block_allocate.argtypes = [P, P, P, P, i32, P, P, P, P, P, i32, i32, i32, P, P, P]
            lib.oracle_block_allocate.restype = ctypes.c_int
            lib.oracle_qrecord_bytes.argtypes = [i32, i32, i32]
            lib.oracle_qrecord_bytes.restype = ctypes.c_size_t
            lib.oracle_kv_quantize_row.argtypes = [P, i32, i32, P, P]
            lib.oracle_kv_quantize_row.restype = ctypes.c_int
            lib.oracle_qcode_offset.argtypes = [i32, i32, i32, i32, i32, i32, P]
            lib.oracle_qcode_offset.restype = ctypes.c_int64
            lib.oracle_paged_kv_append_quant.argtypes = [P, i32, i32, i32, i32, i32, P, i32, P, P, P, P, i32]
            lib.oracle_paged_kv_append_quant.restype = ctypes.c_int
            lib.oracle_qpool_dequant.argtypes = [P, i32, i32, i32, i32, i32, P, P]
            lib.oracle_qpool_dequant.restype = None
            lib.oracle_paged_attention_quant.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, i32, P, i32,
                                                         i32, P, P, i32, P, ctypes.c_double, P, i32]
            lib.oracle_paged_attention_quant.restype = ctypes.c_int
            _lib = lib
        return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_num_threads() -> int:
    return len(os.sched_getaffinity(0))


def paged_kv_append(k_pool, v_pool, block_tables, context_lens_old, new_starts, k_new, v_new):
    """Scatter the new tokens' K/V rows into the pools, in place.

    k_pool/v_pool: uint16 (bf16 bits) [num_blocks, H_kv, block_size, head_dim], C-contiguous.
    block_tables: int32 [S, max_blocks]; context_lens_old: int32 [S];
    new_starts: int32 [S+1]; k_new/v_new: uint16 [R_new, H_kv, head_dim].
    """
    lib = _load()
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    nb, hkv, bs, d = k_pool.shape
    bt = _c(block_tables, np.int32)
    rc = lib.oracle_paged_kv_append(
        _ptr(k_pool), _ptr(v_pool), nb, bs, hkv, d, _ptr(bt), bt.shape[1],
        _ptr(_c(context_lens_old, np.int32)), _ptr(_c(new_starts, np.int32)),
        _ptr(_c(k_new, np.uint16)), _ptr(_c(v_new, np.uint16)), bt.shape[0])
    if rc != 0:
        raise ValueError(f"oracle_paged_kv_append failed with status {rc}")


def paged_attention(k_pool, v_pool, q, q_starts, block_tables, context_lens,
                    kv_head_of_q_head=None, sinks=None, causal=False, scale=None,
                    num_threads=None, tree_masks=None):
    """Float64 attention over the paged pool; returns float64 [R, H_q, head_dim].

    q: uint16 (bf16 bits) [R, H_q, head_dim]; q_starts: int32 [S+1];
    context_lens: int32 [S] (keys in the cache, including any just appended);
    kv_head_of_q_head: int32 [H_q] or None (contiguous groups);
    sinks: float32 [H_q] or None; scale: None means 1/sqrt(head_dim).
    tree_masks: uint32 [R] or None: bit i of row r = row r sees window token i
    (the sequence's last W keys); overrides `causal`.
    """
    lib = _load()
    nb, hkv, bs, d = k_pool.shape
    q = _c(q, np.uint16)
    r, hq, dq = q.shape
    assert dq == d
    bt = _c(block_tables, np.int32)
    qs = _c(q_starts, np.int32)
    cl = _c(context_lens, np.int32)
    hm = None if kv_head_of_q_head is None else _c(kv_head_of_q_head, np.int32)
    sk = None if sinks is None else _c(sinks, np.float32)
    tm = None if tree_masks is None else _c(tree_masks, np.uint32)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((r, hq, d), dtype=np.float64)
    rc = lib.oracle_paged_attention(
        _ptr(_c(k_pool, np.uint16)), _ptr(_c(v_pool, np.uint16)), nb, bs, hkv, d,
        _ptr(q), _ptr(qs), _ptr(bt), bt.shape[1], _ptr(cl), cl.shape[0], hq, _ptr(hm),
        _ptr(sk), int(bool(causal)), _ptr(tm), float(scale), _ptr(out),
        int(num_threads or default_num_threads()))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention failed with status {rc}")
    return out


def argmax_rows(logits):
    """Per-row argmax with ties to the lowest index; int32 [rows]."""
    lib = _load()
    lg = _c(logits, np.float32)
    rows, vocab = lg.shape
    out = np.empty(rows, dtype=np.int32)
    lib.oracle_argmax_rows(_ptr(lg), rows, vocab, _ptr(out))
    return out


def spec_accept_greedy(logits, q_starts, draft_tokens):
    """Greedy accept: returns (argmax [R], accept_len [S], out_tokens [R]), all int32."""
    lib = _load()
    lg = _c(logits, np.float32)
    rows, vocab = lg.shape
    qs = _c(q_starts, np.int32)
    dr = _c(draft_tokens, np.int32)
    s = qs.shape[0] - 1
    assert qs[-1] == rows and dr.shape[0] == rows
    am = np.empty(rows, dtype=np.int32)
    al = np.empty(s, dtype=np.int32)
    ot = np.empty(rows, dtype=np.int32)
    lib.oracle_spec_accept_greedy(_ptr(lg), vocab, _ptr(qs), _ptr(dr), s, _ptr(am), _ptr(al), _ptr(ot))
    return am, al, ot


def spec_accept_tree_greedy(logits, q_starts, draft_tokens, parents):
    """Greedy accept over draft trees: returns (argmax [R], accept_len [S], out_tokens [R],
    accepted_rows [R]), all int32.  parents[r]: parent node index of row r within its
    sequence (row 0 of each sequence is the root; its entry is ignored)."""
    lib = _load()
    lg = _c(logits, np.float32)
    rows, vocab = lg.shape
    qs = _c(q_starts, np.int32)
    dr = _c(draft_tokens, np.int32)
    pa = _c(parents, np.int32)
    s = qs.shape[0] - 1
    am = np.empty(rows, dtype=np.int32)
    al = np.empty(s, dtype=np.int32)
    ot = np.empty(rows, dtype=np.int32)
    ar = np.empty(rows, dtype=np.int32)
    rc = lib.oracle_spec_accept_tree_greedy(_ptr(lg), vocab, _ptr(qs), _ptr(dr), _ptr(pa), s, _ptr(am),
                                            _ptr(al), _ptr(ot), _ptr(ar))
    if rc != 0:
        raise ValueError(f"oracle_spec_accept_tree_greedy failed with status {rc}")
    return am, al, ot, ar


def philox4x32_10(counter, key):
    """Philox4x32-10 of a 4-word counter and 2-word key; returns 4 uint32 words."""
    lib = _load()
    c = _c(counter, np.uint32)
    k = _c(key, np.uint32)
    out = np.empty(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def keyed_log(x):
    """The sampler's float32 natural logarithm (fixed float32 operation sequence)."""
    return np.float32(_load().oracle_keyed_log(float(x)))


def spec_accept_sampled(logits, q_starts, draft_tokens, positions, seed, temperature, min_p=0.0,
                        parents=None, top_k=0, top_p=1.0):
    """Sampled (keyed) accept: returns (sampled [R], accept_len [S], out_tokens [R],
    accepted_rows [R]), all int32.  parents None means chains; top_k <= 0 and
    top_p >= 1 switch those filters off."""
    lib = _load()
    lg = _c(logits, np.float32)
    rows, vocab = lg.shape
    qs = _c(q_starts, np.int32)
    dr = _c(draft_tokens, np.int32)
    po = _c(positions, np.int32)
    pa = None if parents is None else _c(parents, np.int32)
    s = qs.shape[0] - 1
    sm = np.empty(rows, dtype=np.int32)
    al = np.empty(s, dtype=np.int32)
    ot = np.empty(rows, dtype=np.int32)
    ar = np.empty(rows, dtype=np.int32)
    rc = lib.oracle_spec_accept_sampled(_ptr(lg), vocab, _ptr(qs), _ptr(dr), _ptr(pa), _ptr(po), int(seed),
                                        float(temperature), int(top_k), float(top_p), float(min_p), s, _ptr(sm),
                                        _ptr(al), _ptr(ot), _ptr(ar))
    if rc != 0:
        raise ValueError(f"oracle_spec_accept_sampled failed with status {rc}")
    return sm, al, ot, ar


def topp_threshold(p_fix: int, total: int) -> int:
    """ceil(p_fix * total / 2^32): the weight a top-p prefix must reach."""
    return int(_load().oracle_topp_threshold(int(p_fix), int(total)))


def keyed_uniform_bits(seed: int, pos: int, v: int) -> int:
    """The 23-bit uniform code the keyed sampler gives token v at position pos under seed."""
    return int(_load().oracle_keyed_uniform_bits(int(seed), int(pos), int(v)))


def keyed_gumbel(seed: int, pos: int, v: int) -> float:
    """Keyed Gumbel noise g = -log(-log(u)) of token v at position pos under seed (float32)."""
    return float(_load().oracle_keyed_gumbel(int(seed), int(pos), int(v)))


def keyed_exp2(y: float) -> float:
    """The fixed float32 2^y (y <= 0) the top-p weights are built from."""
    return float(_load().oracle_keyed_exp2(float(y)))


def topkp_kept(row, temperature, top_k=0, top_p=1.0):
    """(n, order): the top-k / top-p filters keep the first n tokens of `order`
    (logit descending, id ascending)."""
    r = _c(row, np.float32)
    order = np.empty(r.shape[0], dtype=np.int32)
    n = _load().oracle_topkp_kept(_ptr(r), r.shape[0], float(temperature), int(top_k), float(top_p), _ptr(order))
    if n < 0:
        raise MemoryError("oracle_topkp_kept")
    return int(n), order


def fnv1a64(data: bytes) -> int:
    buf = np.frombuffer(bytes(data), dtype=np.uint8) if len(data) else np.zeros(1, np.uint8)
    return int(_load().oracle_fnv1a64(_ptr(np.ascontiguousarray(buf)), len(data)))


def splitmix64_mix(z: int) -> int:
    return int(_load().oracle_splitmix64_mix(z & 0xFFFFFFFFFFFFFFFF))


def block_hashes(tokens, token_starts, block_size, seed, max_blocks_per_seq, chain_in=None):
    """Chained keys of every full block: uint64 [S, max_blocks_per_seq] (0 past the full blocks)."""
    lib = _load()
    tk = _c(tokens, np.int32)
    ts = _c(token_starts, np.int32)
    s = ts.shape[0] - 1
    ci = None if chain_in is None else _c(chain_in, np.uint64)
    out = np.empty((s, max_blocks_per_seq), dtype=np.uint64)
    rc = lib.oracle_block_hashes(_ptr(tk), _ptr(ts), s, int(block_size), int(seed),
                                 None if ci is None else _ptr(ci), _ptr(out), int(max_blocks_per_seq))
    if rc != 0:
        raise ValueError(f"oracle_block_hashes failed with status {rc}")
    return out


# ------------------------------------------------------ quantised KV blocks --
class BlockIndex:
    """The prefix-sharing index of the block allocator as a plain list of entries:
    keys uint64 [n], ids int32 [n] (-1: a key whose allocation failed), refs int32 [n]."""

    def __init__(self, keys=(), ids=(), refs=()):
        self.keys = np.asarray(keys, np.uint64).copy()
        self.ids = np.asarray(ids, np.int32).copy()
        self.refs = np.asarray(refs, np.int32).copy()

    def as_dict(self):
        return {int(k): (int(i), int(r)) for k, i, r in zip(self.keys, self.ids, self.refs)}


def block_allocate(index: BlockIndex, free_ids, free_count: int, block_keys, context_lens, first_block,
                   block_size: int, block_tables):
    """Sequential block allocation with prefix sharing (see oracle_block_allocate).

    block_keys uint64 [S, max_blocks]; block_tables int32 [S, max_blocks] (entries before
    first_block are kept).  Returns (new BlockIndex, block_tables, fresh int32 [S, max_blocks],
    free_count, status_bits)."""
    lib = _load()
    keys = _c(block_keys, np.uint64)
    S, mb = keys.shape
    tables = _c(block_tables, np.int32).copy()
    fresh = np.zeros((S, mb), np.int32)
    n0 = len(index.keys)
    cap = n0 + S * mb + 1
    ik = np.zeros(cap, np.uint64)
    ii = np.zeros(cap, np.int32)
    ir = np.zeros(cap, np.int32)
    ik[:n0], ii[:n0], ir[:n0] = index.keys, index.ids, index.refs
    n = np.array([n0], np.int32)
    fc = np.array([free_count], np.int32)
    bits = np.zeros(1, np.int32)
    fids = _c(free_ids, np.int32)
    rc = lib.oracle_block_allocate(_ptr(ik), _ptr(ii), _ptr(ir), _ptr(n), cap, _ptr(fids), _ptr(fc), _ptr(keys),
                                   _ptr(_c(context_lens, np.int32)), _ptr(_c(first_block, np.int32)), S,
                                   int(block_size), mb, _ptr(tables), _ptr(fresh), _ptr(bits))
    if rc != 0:
        raise RuntimeError("oracle_block_allocate failed")
    k = int(n[0])
    return BlockIndex(ik[:k], ii[:k], ir[:k]), tables, fresh, int(fc[0]), int(bits[0])


def qrecord_bytes(block_size, head_dim, bits) -> int:
    """Bytes of one (block, KV head) record of the quantised pool."""
    return int(_load().oracle_qrecord_bytes(int(block_size), int(head_dim), int(bits)))


def kv_quantize_row(x_bits, bits):
    """Quantise one bf16 row (uint16 bits [d]); returns (codes int32 [d], scale float32)."""
    x = _c(x_bits, np.uint16)
    codes = np.empty(x.shape[0], dtype=np.int32)
    scale = np.zeros(1, dtype=np.float32)
    rc = _load().oracle_kv_quantize_row(_ptr(x), x.shape[0], int(bits), _ptr(codes), _ptr(scale))
    if rc != 0:
        raise ValueError(f"oracle_kv_quantize_row failed with status {rc}")
    return codes, scale[0]


def qcode_offset(sec, t, i, head_dim, block_size, bits):
    """(byte offset, bit shift) of the code of (section 0=K / 1=V, slot t, dim i) in a record."""
    sh = ctypes.c_int32(0)
    off = _load().oracle_qcode_offset(int(sec), int(t), int(i), int(head_dim), int(block_size), int(bits),
                                      ctypes.byref(sh))
    return int(off), int(sh.value)


def new_qpool(num_blocks, num_kv_heads, block_size, head_dim, bits, fill=None):
    """A record pool uint8 [num_blocks, H_kv, record_bytes] (zeros, or the given fill bytes)."""
    rb = qrecord_bytes(block_size, head_dim, bits)
    pool = np.zeros((num_blocks, num_kv_heads, rb), dtype=np.uint8)
    if fill is not None:
        pool[...] = fill
    return pool


def paged_kv_append_quant(records, block_size, head_dim, bits, block_tables, context_lens_old, new_starts,
                          k_new, v_new):
    """Quantise the new tokens' K/V rows into the record pool, in place."""
    lib = _load()
    assert records.dtype == np.uint8 and records.flags.c_contiguous
    nb, hkv, rb = records.shape
    assert rb == qrecord_bytes(block_size, head_dim, bits)
    bt = _c(block_tables, np.int32)
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    rc = lib.oracle_paged_kv_append_quant(_ptr(records), nb, int(block_size), hkv, int(head_dim), int(bits),
                                          _ptr(bt), bt.shape[1], _ptr(_c(context_lens_old, np.int32)),
                                          _ptr(_c(new_starts, np.int32)), _ptr(kn), _ptr(vn),
                                          len(context_lens_old))
    if rc != 0:
        raise ValueError(f"oracle_paged_kv_append_quant failed with status {rc}")


def qpool_dequant(records, block_size, head_dim, bits):
    """Every record read back: float64 K, V [num_blocks, H_kv, block_size, head_dim]."""
    rec = _c(records, np.uint8)
    nb, hkv, _ = rec.shape
    k = np.empty((nb, hkv, block_size, head_dim), dtype=np.float64)
    v = np.empty_like(k)
    _load().oracle_qpool_dequant(_ptr(rec), nb, int(block_size), hkv, int(head_dim), int(bits), _ptr(k), _ptr(v))
    return k, v


def paged_attention_quant(records, block_size, head_dim, bits, q, q_starts, block_tables, context_lens,
                          kv_head_of_q_head=None, sinks=None, causal=False, scale=None, num_threads=None,
                          tree_masks=None):
    """paged_attention over the quantised record pool (K, V read back as code * scale)."""
    lib = _load()
    rec = _c(records, np.uint8)
    nb, hkv, _ = rec.shape
    q = _c(q, np.uint16)
    r, hq, dq = q.shape
    assert dq == head_dim
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    hm = None if kv_head_of_q_head is None else _c(kv_head_of_q_head, np.int32)
    sk = None if sinks is None else _c(sinks, np.float32)
    tm = None if tree_masks is None else _c(tree_masks, np.uint32)
    if scale is None:
        scale = 1.0 / np.sqrt(head_dim)
    out = np.zeros((r, hq, head_dim), dtype=np.float64)
    rc = lib.oracle_paged_attention_quant(
        _ptr(rec), int(bits), nb, int(block_size), hkv, int(head_dim), _ptr(q), _ptr(_c(q_starts, np.int32)),
        _ptr(bt), bt.shape[1], _ptr(cl), cl.shape[0], hq, _ptr(hm), _ptr(sk), int(bool(causal)), _ptr(tm),
        float(scale), _ptr(out), int(num_threads or default_num_threads()))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention_quant failed with status {rc}")
    return out


def paged_attention_sparse(k_pool, v_pool, q, q_starts, block_tables, context_lens, key_idx, key_counts,
                           kv_head_of_q_head=None, sinks=None, scale=None):
    """Attention of every row over its own list of key positions: float64 [R, H_q, D].

    key_idx int32 [R, max_keys] (positions within the row's sequence), key_counts int32 [R]."""
    lib = _load()
    nb, hkv, bs, d = k_pool.shape
    q = _c(q, np.uint16)
    r, hq, dq = q.shape
    assert dq == d
    bt = _c(block_tables, np.int32)
    ki = _c(key_idx, np.int32)
    kc = _c(key_counts, np.int32)
    hm = None if kv_head_of_q_head is None else _c(kv_head_of_q_head, np.int32)
    sk = None if sinks is None else _c(sinks, np.float32)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((r, hq, d), dtype=np.float64)
    rc = lib.oracle_paged_attention_sparse(
        _ptr(_c(k_pool, np.uint16)), _ptr(_c(v_pool, np.uint16)), nb, bs, hkv, d, _ptr(q),
        _ptr(_c(q_starts, np.int32)), _ptr(bt), bt.shape[1], _ptr(_c(context_lens, np.int32)),
        len(context_lens), _ptr(ki), _ptr(kc), ki.shape[1] if ki.ndim == 2 else 0, hq, _ptr(hm), _ptr(sk),
        float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention_sparse failed with status {rc}")
    return out
