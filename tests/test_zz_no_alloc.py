"""The allocation-free attention entry point, called through the C ABI.

paged_attention_forward_noalloc serves callers that cannot allocate device memory
(a stream being captured into a graph that must not allocate, runtimes that own
all device memory through their own arena, plug-in hosts whose allocator the
library cannot reach).  It keeps its workspace in a fixed array inside the
library.  These checks compare it with paged_attention_forward (caller-provided
workspace) on the same inputs, two calls in a row, and check that sizes past the
array's capacity are refused before anything runs.  This file is collected last
so that a stop-at-first-failure run has already run every other test.
"""
import ctypes

import numpy as np
import pytest

from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import TOL_MAX, TOL_MEAN, gpu_batch

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


@pytest.mark.parametrize("name,num_seqs", [("tiny_decode", None), ("cb_mix", 16), ("sinks_scale", 8),
                                           ("spec_verify", 3)])
def test_noalloc_matches_workspace_entry_point_twice(pkv, name, num_seqs):
    b = wl.make_workload(name, seed=21, num_seqs=num_seqs)
    g = gpu_batch(b)
    if b.new_starts[-1] > 0:
        pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"],
                            g["new_starts"], g["k_new"], g["v_new"])
    ref = pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                      g["context_lens"], max_context_len=b.max_context_len,
                                      max_q_rows_per_seq=b.max_q_rows_per_seq, sinks=g["sinks"],
                                      causal=b.causal).float().cpu().numpy()
    for call in range(2):
        out = torch.full_like(g["q"], float("nan"))
        rc = _noalloc(pkv, g, b, out)
        assert rc == 0, pkv.lib().pkv_last_error_string()
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        err = np.abs(got - ref)
        assert np.all(np.isfinite(got)), f"call {call}: unwritten output"
        assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, f"call {call}: max {err.max()}"
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
