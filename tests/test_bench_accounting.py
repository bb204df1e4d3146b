"""bench.py's algorithmic accounting, checked against brute-force counts on small batches.

The roofline divides these counts by measured time, so a wrong count would misstate every
fraction: flops are 4 * head_dim per (row, q head, visible key), bytes count each distinct
K / V token once (shared prefix blocks once).
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_attention_forward_gb300 import workloads as wl  # noqa: E402


def _visible_keys_brute(b):
    n = 0
    for s in range(b.num_seqs):
        W = int(b.q_starts[s + 1] - b.q_starts[s])
        L = int(b.context_lens[s])
        for w in range(W):
            for t in range(L):
                if b.tree_masks is not None:
                    r = int(b.q_starts[s]) + w
                    ok = t < L - W or (int(b.tree_masks[r]) >> (t - (L - W))) & 1
                elif b.causal:
                    ok = t <= L - W + w
                else:
                    ok = True
                n += bool(ok)
    return n


def test_flops_count_visible_keys():
    for causal in (False, True):
        b = wl.build_batch(5, name="acct", lens=np.array([1, 40, 77, 300]), n_new=np.array([1, 4, 16, 9]),
                           q_rows=np.array([1, 4, 16, 9]), num_q_heads=6, num_kv_heads=2, head_dim=64,
                           block_size=16, causal=causal)
        assert bench.algorithmic_flops(b) == 4.0 * 64 * 6 * _visible_keys_brute(b)


def test_flops_count_tree_rows():
    b = wl.make_workload("spec_tree", num_seqs=3)
    assert bench.algorithmic_flops(b) == 4.0 * b.head_dim * b.num_q_heads * _visible_keys_brute(b)


def test_bytes_count_shared_prefix_once():
    b = wl.make_workload("cb_mix", num_seqs=8)
    acct = bench.algorithmic_bytes(b)
    B, H, D = b.block_size, b.num_kv_heads, b.head_dim
    # distinct physical (block, slot) positions the tables name, K and V, every KV head
    slots = set()
    for s in range(b.num_seqs):
        for t in range(int(b.context_lens[s])):
            slots.add((int(b.block_tables[s, t // B]), t % B))
    assert acct["kv_unique"] == len(slots) * H * D * 2 * 2
    assert acct["kv_logical"] == int(b.context_lens.sum()) * H * D * 2 * 2
