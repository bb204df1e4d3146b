"""One decode-and-verify step captured as a CUDA graph replays bit-identically to the eager calls.

The library allocates nothing and keeps no host state across calls (outputs and workspaces are
the caller's), so a serving loop can capture its step once and replay it: append of the verify
window's tokens, causal paged attention and greedy accept, all on the capturing stream.
"""
import numpy as np
import pytest

from paged_kv_attention_forward_gb300 import workloads as wl
from _helpers import dev, gpu_batch, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


def test_captured_step_replays_bit_identically(pkv):
    b = wl.make_workload("spec_verify", seed=5, num_seqs=4)
    g = gpu_batch(b)
    logits, drafts = dev(b.logits), dev(b.draft_tokens)
    R, S, V = b.total_q_rows, b.num_seqs, b.logits.shape[1]
    k0, v0 = g["k_pool"].clone(), g["v_pool"].clone()
    ws = pkv.new_attention_workspace(S, R, b.num_q_heads, b.num_kv_heads, b.head_dim, b.max_context_len, "cuda")
    acc_ws = torch.empty(max(pkv.spec_accept_workspace_size(R, V), 256), dtype=torch.uint8, device="cuda")
    out = torch.empty((R, b.num_q_heads, b.head_dim), dtype=torch.bfloat16, device="cuda")
    am, al, ot = (torch.empty(n, dtype=torch.int32, device="cuda") for n in (R, S, R))

    def step(stream):
        pkv.paged_kv_append(g["k_pool"], g["v_pool"], g["block_tables"], g["context_lens_old"], g["new_starts"],
                            g["k_new"], g["v_new"], stream=stream)
        pkv.paged_attention_forward(g["k_pool"], g["v_pool"], g["q"], g["q_starts"], g["block_tables"],
                                    g["context_lens"], max_context_len=b.max_context_len,
                                    max_q_rows_per_seq=b.max_q_rows_per_seq, causal=True, out=out,
                                    workspace=ws, stream=stream)
        pkv.spec_accept_greedy(logits, g["q_starts"], drafts, argmax_out=am, accept_len=al, out_tokens=ot,
                               workspace=acc_ws, stream=stream)

    def snapshot():
        torch.cuda.synchronize()
        return [host_bits(g["k_pool"]), host_bits(g["v_pool"]), host_bits(out)] + \
               [t.cpu().numpy().copy() for t in (am, al, ot)]

    step(torch.cuda.current_stream())
    eager = snapshot()

    g["k_pool"].copy_(k0)
    g["v_pool"].copy_(v0)
    out.zero_()
    for t in (am, al, ot):
        t.fill_(-7)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    for _ in range(2):   # the append rewrites the same slots, so every replay gives the same bytes
        graph.replay()
        got = snapshot()
        for e, r in zip(eager, got):
            assert np.array_equal(e, r)
    rc, bits = pkv.device_status()
    assert rc == 0 and bits == 0
