"""The allocation-free attention entry point, called through the C ABI.

paged_attention_forward_noalloc serves callers that cannot allocate device memory
(a stream being captured into a graph that must not allocate, runtimes that own
all device memory through their own arena, plug-in hosts whose allocator the
library cannot reach).  It keeps its workspace in a fixed array inside the
library.  Both entry points launch the same kernels on the same inputs, so these
checks require the allocation-free output to equal paged_attention_forward's
(caller-provided workspace) bit for bit, on two calls in a row and after a larger
shape has left its partials in the array, and to match the float64 oracle within
the attention tolerance; sizes past the array's capacity must be refused before
anything runs.  This file is collected last
so that a stop-at-first-failure run has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import assert_close_to_oracle, gpu_batch, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


def _noalloc(pkv, g, b, out):
    pool = pkv._Pool(g["k_pool"].data_ptr(), g["v_pool"].data_ptr(), b.num_blocks, b.block_size,
                     b.num_kv_heads, b.head_dim)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return pkv.lib().paged_attention_forward_noalloc(
        ctypes.byref(pool), p(g["q"]), p(g["q_starts"]), p(g["block_tables"]), b.max_blocks_per_seq,
        p(g["context_lens"]), b.num_seqs, b.total_q_rows, b.max_context_len, b.max_q_rows_per_seq,
        b.num_q_heads, None, p(g["sinks"]), int(b.causal), 0.0, p(out), pkv.PKV_DTYPE_BF16, stream)


def _workspace_path(pkv, g, b):
    if b.new_starts[-1] > 0:
        pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"],
                            g["new_starts"], g["k_new"], g["v_new"])
    out = pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                      g["context_lens"], max_context_len=b.max_context_len,
                                      max_q_rows_per_seq=b.max_q_rows_per_seq, sinks=g["sinks"],
                                      causal=b.causal)
    torch.cuda.synchronize()
    return out


def _oracle(b):
    k, v = b.k_pool[0].copy(), b.v_pool[0].copy()
    if b.new_starts[-1] > 0:
        oracle.paged_kv_append(k, v, b.block_tables, b.context_lens_old, b.new_starts, b.k_new[0], b.v_new[0])
    return oracle.paged_attention(k, v, b.q[0], b.q_starts, b.block_tables, b.context_lens, sinks=b.sinks,
                                  causal=b.causal)


# The largest shape runs first, so that the shared array still holds its partials (more
# rows and more splits) when the smaller shapes run after it: a stale partial that leaked
# into a later result would change its bits.
CASES = [("cb_mix", 16), ("spec_verify", 3), ("sinks_scale", 8), ("tiny_decode", None)]


def test_noalloc_is_bit_identical_to_the_workspace_entry_point_twice(pkv):
    for name, num_seqs in CASES:
        b = wl.make_workload(name, seed=21, num_seqs=num_seqs)
        g = gpu_batch(b)
        ref_bits = host_bits(_workspace_path(pkv, g, b))
        for call in range(2):
            out = torch.full_like(g["q"], float("nan"))
            rc = _noalloc(pkv, g, b, out)
            assert rc == 0, pkv.lib().pkv_last_error_string()
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(out), ref_bits), f"{name}, call {call}: differs from the workspace path"
        # and both against the float64 oracle, within the attention tolerance
        assert_close_to_oracle(out.float().cpu().numpy(), _oracle(b), what=f"{name} (allocation-free)")
        rc, bits = pkv.device_status()
        assert rc == 0 and bits == 0


def test_noalloc_refuses_sizes_past_its_scratch(pkv):
    b = wl.make_workload("tiny_decode", seed=22)
    g = gpu_batch(b)
    big = 1 << 22                                    # a context bound whose partials cannot fit
    tables = torch.zeros((b.num_seqs, big // b.block_size), dtype=torch.int32, device="cuda")
    g = dict(g, block_tables=tables)
    b.block_tables = np.zeros((b.num_seqs, big // b.block_size), np.int32)
    out = torch.empty_like(g["q"])
    pool = pkv._Pool(g["k_pool"].data_ptr(), g["v_pool"].data_ptr(), b.num_blocks, b.block_size,
                     b.num_kv_heads, b.head_dim)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = pkv.lib().paged_attention_forward_noalloc(
        ctypes.byref(pool), p(g["q"]), p(g["q_starts"]), p(tables), tables.shape[1], p(g["context_lens"]),
        b.num_seqs, b.total_q_rows, big, 1, b.num_q_heads, None, None, 0, 0.0, p(out),
        pkv.PKV_DTYPE_BF16, None)
    assert rc == -4
    assert b"built-in scratch holds" in pkv.lib().pkv_last_error_string()
